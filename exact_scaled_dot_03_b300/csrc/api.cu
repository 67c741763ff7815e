// Host side of the C ABI declared in include/attn.h: argument validation,
// TMA tensor-map encoding, launch configuration and the device status word.
// Everything the caller asks for runs in the kernels of fwd_kernel.cuh and
// decode_kernel.cuh; there is no host or library fallback.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "attn.h"
#include "decode_kernel.cuh"
#include "fwd_kernel.cuh"
#include "rope_kernel.cuh"
#include "bwd_kernel.cuh"

namespace {

using namespace attn_dev;

// Per-device status word: {flags, wait site, block index, unused}.
__device__ unsigned g_attn_status[4];

constexpr int kMaxDevices = 64;

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}

// Per-device values looked up once. Host threads may make their first calls
// concurrently: the slots are atomics, and a lookup that two threads both make
// stores the same value.
unsigned* status_ptr(int dev) {
  static std::atomic<unsigned*> ptrs[kMaxDevices];
  unsigned* p = ptrs[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_attn_status) != cudaSuccess || a == nullptr) return nullptr;
    p = static_cast<unsigned*>(a);
    ptrs[dev].store(p, std::memory_order_release);
  }
  return p;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// A [rows_outer, n, d] bf16 tensor viewed as a 3-D TMA map with a
// {64 columns, box_rows rows, 1} box and 128-byte swizzle. Rows past n read
// as zeros.
bool make_map(CUtensorMap* map, const void* base, int d, long long n, long long outer, int box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(n), static_cast<cuuint64_t>(outer)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(n) * d * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Raises a kernel's dynamic shared-memory limit once per device (setting it
// twice from racing threads is harmless).
using DevFlags = std::atomic<bool>[kMaxDevices];
template <typename K>
bool ensure_smem(K kernel, int bytes, int dev, DevFlags& done) {
  if (done[dev].load(std::memory_order_acquire)) return true;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return false;
  done[dev].store(true, std::memory_order_release);
  return true;
}

// Failure-detection test hook (attn_test_arm_stall): the kind of the kernel
// whose next launch makes one wait stall, or 0.
std::atomic<int> g_armed_stall{0};

// 1 if the hook is armed for `kind` (and disarms it), else 0.
int take_stall(int kind) {
  int expected = kind;
  return g_armed_stall.compare_exchange_strong(expected, 0) ? 1 : 0;
}

// o = 0 and lse = -inf for rows that see no key at all.
__global__ void fill_empty_kernel(__nv_bfloat16* o, float* lse, size_t rows, int d) {
  const size_t n = rows * static_cast<size_t>(d);
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    o[i] = __float2bfloat16_rn(0.f);
    if (lse != nullptr && i % d == 0) lse[i / d] = -CUDART_INF_F;
  }
}

template <int D>
attn_status launch_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                       int Nq, int Nk, float scale, int causal, int window, cudaStream_t stream, int dev,
                       const float2* rope_cs = nullptr, int rope_pmin = 0, int rope_T = 0) {
  static DevFlags smem_set;
  using C = FwdCfg<D>;
  CUtensorMap tq, tk, tv;
  if (!make_map(&tq, q, D, Nq, static_cast<long long>(B) * Hq, 128) ||
      !make_map(&tk, k, D, Nk, static_cast<long long>(B) * Hkv, 128) ||
      !make_map(&tv, v, D, Nk, static_cast<long long>(B) * Hkv, 128))
    return ATTN_ERR_CUDA;
  static DevFlags smem_set_w;
  if (!ensure_smem(attn_fwd_kernel<D, false>, C::SMEM_BYTES, dev, smem_set) ||
      !ensure_smem(attn_fwd_kernel<D, true>, C::SMEM_BYTES, dev, smem_set_w))
    return ATTN_ERR_CUDA;
  FwdArgs a;
  a.o = static_cast<__nv_bfloat16*>(o);
  a.lse = lse;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Nq = Nq;
  a.Nk = Nk;
  a.group = Hq / Hkv;
  a.causal = causal;
  a.causal_offset = Nk - Nq;
  a.window = window;
  a.rope_cs = rope_cs;
  a.rope_pmin = rope_pmin;
  a.rope_T = rope_T;
  a.num_pairs = (Nq + 255) / 256;
  a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  a.status = status_ptr(dev);
  if (a.status == nullptr) return ATTN_ERR_CUDA;
  a.stall = take_stall(ATTN_TEST_STALL_PREFILL);
  dim3 grid(Hq, a.num_pairs, B);
  if (window > 0)
    attn_fwd_kernel<D, true><<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(tq, tk, tv, a);
  else
    attn_fwd_kernel<D, false><<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(tq, tk, tv, a);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

struct DecodePlan {
  int G, GC, qgroups, units, slots;
  size_t part_o_off, part_lse_off, ticket_off, total;
};

// Keys per decode tile and the minimum chunk (in tiles) a CTA takes; both
// must match DecCfg in decode_kernel.cuh.
constexpr int kDecTile = 128;
constexpr int kDecMinChunk = 4;

bool plan_decode(int B, int Hq, int Hkv, int Lmax, int d, DecodePlan* p) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Lmax < 1 || Hq % Hkv != 0) return false;
  if (d != 64 && d != 128) return false;
  p->G = Hq / Hkv;
  p->GC = p->G % 8 == 0 ? 8 : p->G % 4 == 0 ? 4 : p->G % 2 == 0 ? 2 : 1;
  p->qgroups = p->G / p->GC;
  const long long units = static_cast<long long>(B) * Hkv * p->qgroups;
  if (units > (1 << 24)) return false;
  p->units = static_cast<int>(units);
  // A unit of n tiles is cut into at most ceil(n / chunk) + 1 pieces, and a
  // chunk is never shorter than kDecMinChunk tiles.
  const long long tiles = (static_cast<long long>(Lmax) + kDecTile - 1) / kDecTile;
  p->slots = static_cast<int>((tiles + kDecMinChunk - 1) / kDecMinChunk + 1);
  const size_t slots = static_cast<size_t>(p->units) * p->slots * p->GC;
  p->part_o_off = 0;
  p->part_lse_off = slots * d * sizeof(float);
  p->ticket_off = p->part_lse_off + ((slots * sizeof(float) + 15) & ~size_t(15));
  p->total = p->ticket_off + ((static_cast<size_t>(p->units) * sizeof(int) + 15) & ~size_t(15));
  return true;
}

int sm_count(int dev) {
  static std::atomic<int> counts[kMaxDevices];
  int n = counts[dev].load(std::memory_order_acquire);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 0;
    counts[dev].store(n, std::memory_order_release);
  }
  return n;
}

// Paged-cache layout and fused append for a decode launch (all null/zero for
// a contiguous cache without append).
struct DecodePaging {
  const int32_t* block_table = nullptr;
  int bt_stride = 0, page_size = 0, num_pages = 0;
  const void* k_new = nullptr;
  const void* v_new = nullptr;
};

template <int D, int GC>
attn_status launch_decode(const void* q, const void* kc, const void* vc, const int32_t* seqlens, void* o,
                          float* lse, int B, int Hq, int Hkv, int Lmax, float scale, void* ws,
                          const DecodePlan& plan, cudaStream_t stream, int dev, const DecodePaging& pg) {
  static DevFlags smem_set;
  using C = DecCfg<D, GC>;
  CUtensorMap tk, tv, tk16, tv16;  // 16-row boxes: the partial last tile of a contiguous cache
  if (pg.block_table == nullptr) {
    if (!make_map(&tk, kc, D, Lmax, static_cast<long long>(B) * Hkv, C::TK) ||
        !make_map(&tv, vc, D, Lmax, static_cast<long long>(B) * Hkv, C::TK) ||
        !make_map(&tk16, kc, D, Lmax, static_cast<long long>(B) * Hkv, 16) ||
        !make_map(&tv16, vc, D, Lmax, static_cast<long long>(B) * Hkv, 16))
      return ATTN_ERR_CUDA;
  } else {
    const int rows = pg.page_size < C::TK ? pg.page_size : C::TK;
    if (!make_map(&tk, kc, D, pg.page_size, static_cast<long long>(pg.num_pages) * Hkv, rows) ||
        !make_map(&tv, vc, D, pg.page_size, static_cast<long long>(pg.num_pages) * Hkv, rows))
      return ATTN_ERR_CUDA;
    tk16 = tk;  // unused by the paged path
    tv16 = tv;
  }
  if (!ensure_smem(attn_decode_kernel<D, GC>, C::SMEM_BYTES, dev, smem_set)) return ATTN_ERR_CUDA;
  DecArgs a;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.seqlens = seqlens;
  a.o = static_cast<__nv_bfloat16*>(o);
  a.lse = lse;
  uint8_t* w = static_cast<uint8_t*>(ws);
  a.part_o = reinterpret_cast<float*>(w + plan.part_o_off);
  a.part_lse = reinterpret_cast<float*>(w + plan.part_lse_off);
  a.tickets = reinterpret_cast<int*>(w + plan.ticket_off);
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Lmax = Lmax;
  a.group = plan.G;
  a.qgroups = plan.qgroups;
  a.slots = plan.slots;
  a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  a.status = status_ptr(dev);
  if (a.status == nullptr) return ATTN_ERR_CUDA;
  a.block_table = pg.block_table;
  a.bt_stride = pg.bt_stride;
  a.page_size = pg.page_size;
  a.num_pages = pg.num_pages;
  a.k_new = static_cast<const __nv_bfloat16*>(pg.k_new);
  a.v_new = static_cast<const __nv_bfloat16*>(pg.v_new);
  a.k_cache = static_cast<__nv_bfloat16*>(const_cast<void*>(kc));
  a.v_cache = static_cast<__nv_bfloat16*>(const_cast<void*>(vc));
  a.stall = take_stall(ATTN_TEST_STALL_DECODE);
  static_assert(C::TK == kDecTile && C::MIN_CHUNK == kDecMinChunk, "decode plan and kernel disagree");
  const int grid = sm_count(dev);  // persistent: one CTA per SM
  if (grid == 0) return ATTN_ERR_CUDA;
  attn_decode_kernel<D, GC><<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(tk, tv, tk16, tv16, a);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

template <int D>
attn_status dispatch_decode_gc(const void* q, const void* kc, const void* vc, const int32_t* seqlens, void* o,
                               float* lse, int B, int Hq, int Hkv, int Lmax, float scale, void* ws,
                               const DecodePlan& plan, cudaStream_t stream, int dev,
                               const DecodePaging& pg = DecodePaging()) {
  switch (plan.GC) {
    case 8: return launch_decode<D, 8>(q, kc, vc, seqlens, o, lse, B, Hq, Hkv, Lmax, scale, ws, plan, stream, dev, pg);
    case 4: return launch_decode<D, 4>(q, kc, vc, seqlens, o, lse, B, Hq, Hkv, Lmax, scale, ws, plan, stream, dev, pg);
    case 2: return launch_decode<D, 2>(q, kc, vc, seqlens, o, lse, B, Hq, Hkv, Lmax, scale, ws, plan, stream, dev, pg);
    default: return launch_decode<D, 1>(q, kc, vc, seqlens, o, lse, B, Hq, Hkv, Lmax, scale, ws, plan, stream, dev, pg);
  }
}

}  // namespace

namespace {
// Backward workspace, per query row (each head padded to 128 rows): lse2 and Dl
// (fp32, two arrays), then the dK/dV kernel's seed operands (32 bytes per row
// and array, 4 KiB per 128-row tile).
bool plan_bwd(int B, int Hq, int Nq, int* Nq_pad, size_t* bytes) {
  if (B < 1 || Hq < 1 || Nq < 0) return false;
  *Nq_pad = (Nq + 127) / 128 * 128;
  *bytes = static_cast<size_t>(B) * Hq * static_cast<size_t>(*Nq_pad) * (2 * sizeof(float) + 2 * 32);
  return true;
}

// The dQ kernel runs beside the dK/dV kernel on a library stream of lower
// priority (they share no output): the dK/dV launch keeps the SMs it needs
// for its heaviest key tiles, and dQ CTAs take up SMs as its last wave thins
// out. Created once per device; the mutex keeps each call's fork and join
// (record, wait, launch, record, wait) in one piece when host threads call at
// once.
struct BwdPipe {
  std::mutex mu;
  bool ready = false;
  cudaStream_t s_dq = nullptr;
  cudaEvent_t prep_done = nullptr, dq_done = nullptr;
};
BwdPipe& bwd_pipe(int dev) {
  static BwdPipe pipes[kMaxDevices];
  return pipes[dev];
}
bool bwd_pipe_init(BwdPipe& p) {
  if (p.ready) return true;
  int lowest = 0, highest = 0;
  if (cudaDeviceGetStreamPriorityRange(&lowest, &highest) != cudaSuccess ||
      cudaStreamCreateWithPriority(&p.s_dq, cudaStreamNonBlocking, lowest) != cudaSuccess ||
      cudaEventCreateWithFlags(&p.prep_done, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&p.dq_done, cudaEventDisableTiming) != cudaSuccess)
    return false;
  p.ready = true;
  return true;
}

template <int D>
attn_status launch_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                       void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Nq, int Nk, float scale, int causal,
                       float* ws, int Nq_pad, cudaStream_t s, int dev) {
  using C = BwdCfg<D>;
  static DevFlags smem_kv, smem_q;
  CUtensorMap tq, tk, tv, tdo;
  if (!make_map(&tq, q, D, Nq, static_cast<long long>(B) * Hq, 128) ||
      !make_map(&tdo, dout, D, Nq, static_cast<long long>(B) * Hq, 128) ||
      !make_map(&tk, k, D, Nk, static_cast<long long>(B) * Hkv, 128) ||
      !make_map(&tv, v, D, Nk, static_cast<long long>(B) * Hkv, 128))
    return ATTN_ERR_CUDA;
  if (!ensure_smem(attn_bwd_dkdv_kernel<D>, C::KV_SMEM_BYTES, dev, smem_kv) ||
      !ensure_smem(attn_bwd_dq_kernel<D>, C::Q_SMEM_BYTES, dev, smem_q))
    return ATTN_ERR_CUDA;
  BwdArgs a;
  a.dq = static_cast<__nv_bfloat16*>(dq);
  a.dk = static_cast<__nv_bfloat16*>(dk);
  a.dv = static_cast<__nv_bfloat16*>(dv);
  const long long rows = static_cast<long long>(B) * Hq * Nq_pad;
  a.lse2 = ws;
  a.dl = ws + rows;
  uint8_t* seed_l = reinterpret_cast<uint8_t*>(ws + 2 * rows);
  uint8_t* seed_d = seed_l + rows * 32;
  a.seed_l = seed_l;
  a.seed_d = seed_d;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Nq = Nq;
  a.Nk = Nk;
  a.Nq_pad = Nq_pad;
  a.group = Hq / Hkv;
  a.causal = causal;
  a.causal_offset = Nk - Nq;
  a.scale = scale;
  a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  a.status = status_ptr(dev);
  const int sms = sm_count(dev);
  if (a.status == nullptr || sms == 0) return ATTN_ERR_CUDA;
  a.stall = take_stall(ATTN_TEST_STALL_BACKWARD);
  const long long heads = static_cast<long long>(B) * Hq;
  const long long threads = heads * Nq_pad * (D / 8);
  const int blocks = static_cast<int>(std::min<long long>((threads + 255) / 256, static_cast<long long>(sms) * 16));
  bwd_prep_kernel<D><<<blocks, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(o),
                                            static_cast<const __nv_bfloat16*>(dout), lse, ws, ws + rows, seed_l,
                                            seed_d, scale, heads, Nq, Nq_pad);
  BwdPipe& P = bwd_pipe(dev);
  std::lock_guard<std::mutex> lock(P.mu);
  if (!bwd_pipe_init(P)) return ATTN_ERR_CUDA;
  bool ok = cudaEventRecord(P.prep_done, s) == cudaSuccess;  // both kernels read what the prep kernel wrote
  attn_bwd_dkdv_kernel<D><<<dim3(2 * ((Nk + 127) / 128), (Hkv + 1) / 2, B), C::THREADS, C::KV_SMEM_BYTES, s>>>(
      tq, tk, tv, tdo, a);
  ok = ok && cudaStreamWaitEvent(P.s_dq, P.prep_done, 0) == cudaSuccess;
  if (ok) attn_bwd_dq_kernel<D><<<dim3(Hq, (Nq + 127) / 128, B), C::THREADS, C::Q_SMEM_BYTES, P.s_dq>>>(tq, tk, tv, tdo, a);
  ok = ok && cudaEventRecord(P.dq_done, P.s_dq) == cudaSuccess;
  ok = ok && cudaStreamWaitEvent(s, P.dq_done, 0) == cudaSuccess;  // the call ends on `stream` with both
  return ok && cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}
}  // namespace

extern "C" {

attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                     int Nq, int Nk, int d, float scale, int causal, void* stream) {
  return attn_fwd_window(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, causal, 0, stream);
}

attn_status attn_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                            int Hkv, int Nq, int Nk, int d, float scale, int causal, int window, void* stream) {
  if (window < 0) return ATTN_ERR_INVALID_ARG;
  // k and v may be NULL only when there are no keys (an empty tensor has no storage).
  if (q == nullptr || o == nullptr || (Nk > 0 && (k == nullptr || v == nullptr))) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 0 || Nk < 0 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      (lse != nullptr && !aligned(lse, 4)))
    return ATTN_ERR_INVALID_ARG;  // (NULL is aligned)
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (B > 65535 || (Nq + 255) / 256 > 65535) return ATTN_ERR_UNSUPPORTED;
  if (Nq == 0) return ATTN_OK;
  const int dev = current_device();
  if (dev < 0) return ATTN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (Nk == 0) {
    const size_t rows = static_cast<size_t>(B) * Hq * Nq;
    const int sms = sm_count(dev);
    if (sms == 0) return ATTN_ERR_CUDA;
    const int blocks = static_cast<int>(std::min<size_t>((rows * d + 255) / 256, static_cast<size_t>(sms) * 16));
    fill_empty_kernel<<<blocks, 256, 0, s>>>(static_cast<__nv_bfloat16*>(o), lse, rows, d);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
  }
  if (d == 64) return launch_fwd<64>(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, scale, causal, window, s, dev);
  return launch_fwd<128>(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, scale, causal, window, s, dev);
}

namespace {
// ---------------------------------------------------------------- host-buffer prefill
// Staging in the caller's workspace (every piece 256-byte aligned):
//   kHostKvSlots  x (K, V of one (batch, KV head) group)
//   ATTN_FWD_HOST_SLOTS x (Q, O, LSE of one chunk: up to all G query heads of a group)
constexpr int kHostKvSlots = 2;
struct HostPlan {
  size_t q_bytes, kv_bytes, lse_bytes;  // per query head (q, o, lse) and per group (k, v)
  size_t kv_slot, q_slot, o_off, lse_off, q_base, total;
};
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
bool plan_host(int B, int Hq, int Hkv, int Nq, int Nk, int d, HostPlan* p) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 0 || Nk < 0 || Hq % Hkv != 0 || (d != 64 && d != 128)) return false;
  const size_t G = static_cast<size_t>(Hq / Hkv);
  p->q_bytes = static_cast<size_t>(Nq) * d * 2;
  p->kv_bytes = static_cast<size_t>(Nk) * d * 2;
  p->lse_bytes = static_cast<size_t>(Nq) * 4;
  p->kv_slot = 2 * align256(p->kv_bytes);
  p->o_off = align256(G * p->q_bytes);
  p->lse_off = p->o_off + align256(G * p->q_bytes);
  p->q_slot = p->lse_off + align256(G * p->lse_bytes);
  p->q_base = kHostKvSlots * p->kv_slot;
  p->total = p->q_base + ATTN_FWD_HOST_SLOTS * p->q_slot;
  return true;
}

// Query heads per chunk: the largest divisor of the group size G whose chunk
// still fills about two CTAs per SM (a chunk of heads * ceil(Nq/256) CTAs).
// Smaller chunks shorten the start and end of the pipeline, where only one
// copy direction is busy; G heads (one chunk per group) when even a single
// head has that many CTAs.
int host_heads_per_chunk(int G, int Nq, int sms) {
  const long long pairs = (Nq + 255) / 256;
  const long long target = 2LL * sms;
  int best = 1;
  for (int h = 1; h <= G; ++h)
    if (G % h == 0 && h * pairs <= target) best = h;
  return best;
}

// The copy streams and events of one device, created on its first call.
struct HostPipe {
  std::mutex mu;  // calls on one device queue their work one at a time
  bool ready = false;
  cudaStream_t s_in = nullptr, s_out = nullptr;
  cudaEvent_t entry = nullptr, last = nullptr;
  cudaEvent_t in_done[ATTN_FWD_HOST_SLOTS] = {}, comp_done[ATTN_FWD_HOST_SLOTS] = {},
              out_done[ATTN_FWD_HOST_SLOTS] = {}, kv_free[kHostKvSlots] = {};
};
HostPipe& host_pipe(int dev) {
  static HostPipe pipes[kMaxDevices];
  return pipes[dev];
}
bool host_pipe_init(HostPipe& p) {
  if (p.ready) return true;
  auto ev = [](cudaEvent_t* e) { return cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess; };
  if (cudaStreamCreateWithFlags(&p.s_in, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&p.s_out, cudaStreamNonBlocking) != cudaSuccess || !ev(&p.entry) || !ev(&p.last))
    return false;
  for (int i = 0; i < ATTN_FWD_HOST_SLOTS; ++i)
    if (!ev(&p.in_done[i]) || !ev(&p.comp_done[i]) || !ev(&p.out_done[i])) return false;
  for (int i = 0; i < kHostKvSlots; ++i)
    if (!ev(&p.kv_free[i])) return false;
  p.ready = true;
  return true;
}
}  // namespace

size_t attn_fwd_host_workspace_size(int B, int Hq, int Hkv, int Nq, int Nk, int d) {
  HostPlan p;
  return plan_host(B, Hq, Hkv, Nq, Nk, d, &p) ? p.total : 0;
}

attn_status attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                          int Nq, int Nk, int d, float scale, int causal, void* workspace, size_t workspace_bytes,
                          void* stream) {
  // q, o may be NULL only when there are no queries, k, v only when there are no keys.
  if ((Nq > 0 && (q == nullptr || o == nullptr)) || (Nk > 0 && (k == nullptr || v == nullptr)))
    return ATTN_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 0 || Nk < 0 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (B > 65535 || (Nq + 255) / 256 > 65535) return ATTN_ERR_UNSUPPORTED;
  HostPlan plan;
  if (!plan_host(B, Hq, Hkv, Nq, Nk, d, &plan)) return ATTN_ERR_INVALID_ARG;
  if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < plan.total) return ATTN_ERR_INVALID_ARG;
  if (Nq == 0) return ATTN_OK;
  const int dev = current_device();
  if (dev < 0) return ATTN_ERR_CUDA;
  const int sms = sm_count(dev);
  if (sms == 0) return ATTN_ERR_CUDA;
  HostPipe& P = host_pipe(dev);
  std::lock_guard<std::mutex> lock(P.mu);
  if (!host_pipe_init(P)) return ATTN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int G = Hq / Hkv;
  const int hc = host_heads_per_chunk(G, Nq, sms);  // query heads per chunk
  const int per_group = G / hc;
  const int groups = B * Hkv;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const uint8_t* qh = static_cast<const uint8_t*>(q);
  const uint8_t* kh = static_cast<const uint8_t*>(k);
  const uint8_t* vh = static_cast<const uint8_t*>(v);
  uint8_t* oh = static_cast<uint8_t*>(o);
  uint8_t* lh = reinterpret_cast<uint8_t*>(lse);
  const size_t cq = hc * plan.q_bytes, cl = hc * plan.lse_bytes;  // bytes of one chunk's Q (= O) and LSE
  bool ok = true;
  attn_status st = ATTN_OK;
  auto chk = [&](cudaError_t e) { ok = ok && (e == cudaSuccess); };
  // Nothing starts before the work queued on `stream` up to this call.
  chk(cudaEventRecord(P.entry, s));
  chk(cudaStreamWaitEvent(P.s_in, P.entry, 0));
  chk(cudaStreamWaitEvent(P.s_out, P.entry, 0));
  int c = 0;  // chunk index over the whole call
  for (int grp = 0; grp < groups && ok && st == ATTN_OK; ++grp) {
    // group grp = (batch b, KV head g): its query heads g*G .. g*G+G-1 of batch b are
    // contiguous in Q, O and LSE, so chunk c covers bytes [c*cq, (c+1)*cq) of Q and O.
    const int ks = grp % kHostKvSlots;
    uint8_t* kd = ws + ks * plan.kv_slot;
    uint8_t* vd = kd + align256(plan.kv_bytes);
    if (Nk > 0) {
      // the K/V slot is free once every chunk of group grp - kHostKvSlots has run
      if (grp >= kHostKvSlots) chk(cudaStreamWaitEvent(P.s_in, P.kv_free[ks], 0));
      const size_t ko = static_cast<size_t>(grp) * plan.kv_bytes;
      chk(cudaMemcpyAsync(kd, kh + ko, plan.kv_bytes, cudaMemcpyHostToDevice, P.s_in));
      chk(cudaMemcpyAsync(vd, vh + ko, plan.kv_bytes, cudaMemcpyHostToDevice, P.s_in));
    }
    for (int j = 0; j < per_group && ok; ++j, ++c) {
      const int slot = c % ATTN_FWD_HOST_SLOTS;
      uint8_t* base = ws + plan.q_base + slot * plan.q_slot;
      // copy in: the slot's Q is free once the prefill of chunk c - SLOTS is done
      // (the K/V copies above precede it on the same stream)
      if (c >= ATTN_FWD_HOST_SLOTS) chk(cudaStreamWaitEvent(P.s_in, P.comp_done[slot], 0));
      chk(cudaMemcpyAsync(base, qh + c * cq, cq, cudaMemcpyHostToDevice, P.s_in));
      chk(cudaEventRecord(P.in_done[slot], P.s_in));
      // prefill on `stream`: the slot's O, LSE are free once the copy out of chunk c - SLOTS is done
      chk(cudaStreamWaitEvent(s, P.in_done[slot], 0));
      if (c >= ATTN_FWD_HOST_SLOTS) chk(cudaStreamWaitEvent(s, P.out_done[slot], 0));
      if (!ok) break;
      st = attn_fwd(base, Nk > 0 ? kd : nullptr, Nk > 0 ? vd : nullptr, base + plan.o_off,
                    lse != nullptr ? reinterpret_cast<float*>(base + plan.lse_off) : nullptr, 1, hc, 1, Nq, Nk, d,
                    scale, causal, s);
      if (st != ATTN_OK) break;
      chk(cudaEventRecord(P.comp_done[slot], s));
      if (j == per_group - 1) chk(cudaEventRecord(P.kv_free[ks], s));
      // copy out
      chk(cudaStreamWaitEvent(P.s_out, P.comp_done[slot], 0));
      chk(cudaMemcpyAsync(oh + c * cq, base + plan.o_off, cq, cudaMemcpyDeviceToHost, P.s_out));
      if (lse != nullptr)
        chk(cudaMemcpyAsync(lh + c * cl, base + plan.lse_off, cl, cudaMemcpyDeviceToHost, P.s_out));
      chk(cudaEventRecord(P.out_done[slot], P.s_out));
    }
  }
  // `stream` passes this call once every copy out has landed (and the copy-in
  // stream has finished with the workspace).
  chk(cudaEventRecord(P.last, P.s_out));
  chk(cudaStreamWaitEvent(s, P.last, 0));
  chk(cudaEventRecord(P.last, P.s_in));
  chk(cudaStreamWaitEvent(s, P.last, 0));
  if (st != ATTN_OK) return st;
  return ok ? ATTN_OK : ATTN_ERR_CUDA;
}

namespace {
// RoPE workspace: the rotated K ([B, Hkv, Nk, d] bf16), then the (cos, sin)
// table of positions min(0, Nk - Nq) .. Nk - 1, position-major and pair-major.
struct RopePlan {
  size_t k_bytes, cs_off, cst_off, total;
  int T, pmin;
};
bool plan_rope(int B, int Hkv, int Nq, int Nk, int d, RopePlan* p) {
  if (B < 1 || Hkv < 1 || Nq < 0 || Nk < 1 || (d != 64 && d != 128)) return false;
  p->pmin = Nk - Nq < 0 ? Nk - Nq : 0;
  p->T = Nk - p->pmin;
  p->k_bytes = static_cast<size_t>(B) * Hkv * Nk * d * 2;
  p->cs_off = (p->k_bytes + 255) & ~size_t(255);
  const size_t cs_bytes = static_cast<size_t>(p->T) * (d / 2) * sizeof(float2);
  p->cst_off = (p->cs_off + cs_bytes + 255) & ~size_t(255);
  p->total = p->cst_off + cs_bytes;
  return true;
}
}  // namespace

size_t attn_fwd_rope_workspace_size(int B, int Hkv, int Nq, int Nk, int d) {
  RopePlan p;
  return plan_rope(B, Hkv, Nq, Nk, d, &p) ? p.total : 0;
}

attn_status attn_fwd_rope(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                          int Nq, int Nk, int d, float scale, int causal, int window, float rope_base,
                          void* workspace, size_t workspace_bytes, void* stream) {
  if (!std::isfinite(rope_base) || !(rope_base > 1.f) || workspace == nullptr || !aligned(workspace, 256))
    return ATTN_ERR_INVALID_ARG;
  if (q == nullptr || o == nullptr || k == nullptr || v == nullptr) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 0 || Nk < 1 || Hq % Hkv != 0 || window < 0) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      (lse != nullptr && !aligned(lse, 4)))
    return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (B > 65535 || (Nq + 255) / 256 > 65535) return ATTN_ERR_UNSUPPORTED;
  RopePlan rp;
  if (!plan_rope(B, Hkv, Nq, Nk, d, &rp)) return ATTN_ERR_UNSUPPORTED;
  if (workspace_bytes < rp.total) return ATTN_ERR_INVALID_ARG;
  if (Nq == 0) return ATTN_OK;
  const int dev = current_device();
  if (dev < 0) return ATTN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  __nv_bfloat16* k_rot = reinterpret_cast<__nv_bfloat16*>(ws);
  float2* cs = reinterpret_cast<float2*>(ws + rp.cs_off);
  float2* cs_t = reinterpret_cast<float2*>(ws + rp.cst_off);
  RopeArgs ra;
  ra.cs = cs;
  ra.cs_t = cs_t;
  ra.T = rp.T;
  ra.pmin = rp.pmin;
  for (int i = 0; i < d / 2; ++i) ra.w[i] = std::pow(static_cast<double>(rope_base), -2.0 * i / d);
  const int sms = sm_count(dev);
  if (sms == 0) return ATTN_ERR_CUDA;
  const long long rows = static_cast<long long>(B) * Hkv * Nk;
  if (d == 64) {
    rope_table_kernel<64><<<sms * 4, 256, 0, s>>>(ra);
    rope_k_kernel<64><<<sms * 8, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(k), k_rot, cs, rows, Nk, rp.pmin);
  } else {
    rope_table_kernel<128><<<sms * 4, 256, 0, s>>>(ra);
    rope_k_kernel<128><<<sms * 8, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(k), k_rot, cs, rows, Nk, rp.pmin);
  }
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
  if (d == 64) return launch_fwd<64>(q, k_rot, v, o, lse, B, Hq, Hkv, Nq, Nk, scale, causal, window, s, dev, cs_t, rp.pmin, rp.T);
  return launch_fwd<128>(q, k_rot, v, o, lse, B, Hq, Hkv, Nq, Nk, scale, causal, window, s, dev, cs_t, rp.pmin, rp.T);
}


size_t attn_bwd_workspace_size(int B, int Hq, int Nq) {
  int pad;
  size_t bytes;
  return plan_bwd(B, Hq, Nq, &pad, &bytes) ? bytes : 0;
}

attn_status attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                     void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Nq, int Nk, int d, float scale,
                     int causal, void* workspace, size_t workspace_bytes, void* stream) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 0 || Nk < 0 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  // Tensors with no rows may be NULL (an empty tensor has no storage).
  if (Nq > 0 && (q == nullptr || o == nullptr || lse == nullptr || dout == nullptr || dq == nullptr))
    return ATTN_ERR_INVALID_ARG;
  if (Nk > 0 && (k == nullptr || v == nullptr || dk == nullptr || dv == nullptr)) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(dout, 16) ||
      !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) || !aligned(lse, 4) || !aligned(workspace, 256))
    return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (B > 65535 || (Nq + 127) / 128 > 65535 || Hkv > 65535) return ATTN_ERR_UNSUPPORTED;  // grid y / z limits
  int Nq_pad;
  size_t need;
  if (!plan_bwd(B, Hq, Nq, &Nq_pad, &need)) return ATTN_ERR_INVALID_ARG;
  if (Nq > 0 && Nk > 0 && (workspace == nullptr || workspace_bytes < need)) return ATTN_ERR_INVALID_ARG;
  const int dev = current_device();
  if (dev < 0) return ATTN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (Nq == 0 || Nk == 0) {
    // No query or no key: every gradient that exists is zero.
    const size_t qrows = static_cast<size_t>(B) * Hq * Nq, krows = static_cast<size_t>(B) * Hkv * Nk;
    const int sms = sm_count(dev);
    if (sms == 0) return ATTN_ERR_CUDA;
    const int qb = static_cast<int>(std::min<size_t>((qrows * d + 255) / 256, static_cast<size_t>(sms) * 16));
    const int kb = static_cast<int>(std::min<size_t>((krows * d + 255) / 256, static_cast<size_t>(sms) * 16));
    if (qrows > 0) fill_empty_kernel<<<qb, 256, 0, s>>>(static_cast<__nv_bfloat16*>(dq), nullptr, qrows, d);
    if (krows > 0) {
      fill_empty_kernel<<<kb, 256, 0, s>>>(static_cast<__nv_bfloat16*>(dk), nullptr, krows, d);
      fill_empty_kernel<<<kb, 256, 0, s>>>(static_cast<__nv_bfloat16*>(dv), nullptr, krows, d);
    }
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
  }
  float* ws = static_cast<float*>(workspace);
  if (d == 64)
    return launch_bwd<64>(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Nq, Nk, scale, causal, ws, Nq_pad, s, dev);
  return launch_bwd<128>(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Nq, Nk, scale, causal, ws, Nq_pad, s, dev);
}

size_t attn_decode_workspace_size(int B, int Hq, int Hkv, int Lmax, int d) {
  DecodePlan p;
  return plan_decode(B, Hq, Hkv, Lmax, d, &p) ? p.total : 0;
}

attn_status attn_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* seqlens, void* o,
                        float* lse, int B, int Hq, int Hkv, int Lmax, int d, float scale, void* workspace,
                        size_t workspace_bytes, void* stream) {
  if (q == nullptr || k_cache == nullptr || v_cache == nullptr || seqlens == nullptr || o == nullptr ||
      workspace == nullptr)
    return ATTN_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || Lmax < 1 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(o, 16) ||
      !aligned(workspace, 16) || !aligned(seqlens, 4) || (lse != nullptr && !aligned(lse, 4)))
    return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  DecodePlan plan;
  if (!plan_decode(B, Hq, Hkv, Lmax, d, &plan)) return ATTN_ERR_UNSUPPORTED;
  if (workspace_bytes < plan.total) return ATTN_ERR_INVALID_ARG;
  const int dev = current_device();
  if (dev < 0) return ATTN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (d == 64)
    return dispatch_decode_gc<64>(q, k_cache, v_cache, seqlens, o, lse, B, Hq, Hkv, Lmax, scale, workspace, plan,
                                  s, dev);
  return dispatch_decode_gc<128>(q, k_cache, v_cache, seqlens, o, lse, B, Hq, Hkv, Lmax, scale, workspace, plan, s,
                                 dev);
}

namespace {
bool valid_page_size(int p) { return p >= 8 && ((p % 128 == 0) || (128 % p == 0)) && p <= (1 << 20); }
}  // namespace

size_t attn_decode_paged_workspace_size(int B, int Hq, int Hkv, int max_pages_per_seq, int page_size, int d) {
  if (max_pages_per_seq < 1 || !valid_page_size(page_size)) return 0;
  const long long cap = static_cast<long long>(max_pages_per_seq) * page_size;
  if (cap > (1LL << 30)) return 0;
  DecodePlan p;
  return plan_decode(B, Hq, Hkv, static_cast<int>(cap), d, &p) ? p.total : 0;
}

attn_status attn_decode_paged(const void* q, const void* k_new, const void* v_new, void* k_pages, void* v_pages,
                              const int32_t* block_table, const int32_t* seqlens, void* o, float* lse, int B, int Hq,
                              int Hkv, int num_pages, int page_size, int max_pages_per_seq, int d, float scale,
                              void* workspace, size_t workspace_bytes, void* stream) {
  if (q == nullptr || k_pages == nullptr || v_pages == nullptr || block_table == nullptr || seqlens == nullptr ||
      o == nullptr || workspace == nullptr || ((k_new == nullptr) != (v_new == nullptr)))
    return ATTN_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || num_pages < 1 || max_pages_per_seq < 1 || Hq % Hkv != 0)
    return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(o, 16) ||
      !aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(workspace, 16) || !aligned(block_table, 4) ||
      !aligned(seqlens, 4) || (lse != nullptr && !aligned(lse, 4)))
    return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (!valid_page_size(page_size)) return ATTN_ERR_UNSUPPORTED;
  const long long cap = static_cast<long long>(max_pages_per_seq) * page_size;
  if (cap > (1LL << 30) || static_cast<long long>(num_pages) * Hkv > (1LL << 31) - 1) return ATTN_ERR_UNSUPPORTED;
  DecodePlan plan;
  if (!plan_decode(B, Hq, Hkv, static_cast<int>(cap), d, &plan)) return ATTN_ERR_UNSUPPORTED;
  if (workspace_bytes < plan.total) return ATTN_ERR_INVALID_ARG;
  const int dev = current_device();
  if (dev < 0) return ATTN_ERR_CUDA;
  DecodePaging pg;
  pg.block_table = block_table;
  pg.bt_stride = max_pages_per_seq;
  pg.page_size = page_size;
  pg.num_pages = num_pages;
  pg.k_new = k_new;
  pg.v_new = v_new;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (d == 64)
    return dispatch_decode_gc<64>(q, k_pages, v_pages, seqlens, o, lse, B, Hq, Hkv, static_cast<int>(cap), scale,
                                  workspace, plan, s, dev, pg);
  return dispatch_decode_gc<128>(q, k_pages, v_pages, seqlens, o, lse, B, Hq, Hkv, static_cast<int>(cap), scale,
                                 workspace, plan, s, dev, pg);
}

attn_status attn_device_status(void* stream, unsigned* detail) {
  const int dev = current_device();
  if (dev < 0) return ATTN_ERR_CUDA;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
  unsigned words[4] = {0, 0, 0, 0};
  if (cudaMemcpyFromSymbol(words, g_attn_status, sizeof(words)) != cudaSuccess) return ATTN_ERR_CUDA;
  const unsigned zero[4] = {0, 0, 0, 0};
  if (cudaMemcpyToSymbol(g_attn_status, zero, sizeof(zero)) != cudaSuccess) return ATTN_ERR_CUDA;
  if (detail != nullptr) {
    detail[0] = words[0];
    detail[1] = words[1];
    detail[2] = words[2];
  }
  if (words[0] & kStatusWaitTimeout) return ATTN_ERR_TIMEOUT;
  if (words[0] & (kStatusBadSeqlen | kStatusBadPage)) return ATTN_ERR_DEVICE_ARG;
  return ATTN_OK;
}

const char* attn_status_string(attn_status s) {
  switch (s) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_TIMEOUT: return "device pipeline wait timed out";
    case ATTN_ERR_DEVICE_ARG: return "device saw a sequence length outside [0, Lmax] or a page id outside [0, num_pages)";
  }
  return "unknown status";
}

uint64_t attn_score_bytes(int64_t n, int64_t heads, int bytes_per_score) {
  if (n < 0 || heads < 0 || bytes_per_score < 0) return 0;
  return static_cast<uint64_t>(heads) * static_cast<uint64_t>(n) * static_cast<uint64_t>(n) *
         static_cast<uint64_t>(bytes_per_score);
}

uint64_t attn_kv_cache_bytes(int64_t layers, int64_t n, int64_t h_kv, int64_t d_h, int bytes_per_scalar) {
  if (layers < 0 || n < 0 || h_kv < 0 || d_h < 0 || bytes_per_scalar < 0) return 0;
  return 2ull * static_cast<uint64_t>(layers) * static_cast<uint64_t>(n) * static_cast<uint64_t>(h_kv) *
         static_cast<uint64_t>(d_h) * static_cast<uint64_t>(bytes_per_scalar);
}

const char* attn_version(void) { return "exact-attn-sm103 0.1"; }

attn_status attn_test_arm_stall(int kind) {
  if (kind != 0 && kind != ATTN_TEST_STALL_PREFILL && kind != ATTN_TEST_STALL_DECODE &&
      kind != ATTN_TEST_STALL_BACKWARD)
    return ATTN_ERR_INVALID_ARG;
  g_armed_stall.store(kind);
  return ATTN_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Decode for callers that cannot allocate device memory (see
// attn_decode_noalloc in attn.h). The split-KV scratch that attn_decode takes
// as a caller workspace lives here instead, in one file-scope device array.
// Host code must not hand g_noalloc_scratch itself to a kernel: on the host
// that name is only a stand-in for the symbol, not a device address. The
// address is looked up once per device with cudaGetSymbolAddress.
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[ATTN_NOALLOC_SCRATCH_BYTES];

void* noalloc_scratch_ptr(int dev) {
  static std::atomic<void*> ptrs[kMaxDevices];
  void* p = ptrs[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return nullptr;
    ptrs[dev].store(p, std::memory_order_release);
  }
  return p;
}

}  // namespace

extern "C" attn_status attn_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                           const int32_t* seqlens, void* o, float* lse, int B, int Hq, int Hkv,
                                           int Lmax, int d, float scale, void* stream) {
  if (q == nullptr || k_cache == nullptr || v_cache == nullptr || seqlens == nullptr || o == nullptr)
    return ATTN_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || Lmax < 1 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(o, 16) ||
      !aligned(seqlens, 4) || (lse != nullptr && !aligned(lse, 4)))
    return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  DecodePlan plan;
  if (!plan_decode(B, Hq, Hkv, Lmax, d, &plan)) return ATTN_ERR_UNSUPPORTED;
  if (plan.total > ATTN_NOALLOC_SCRATCH_BYTES) return ATTN_ERR_UNSUPPORTED;  // does not fit the static scratch
  const int dev = current_device();
  if (dev < 0) return ATTN_ERR_CUDA;
  void* scratch = noalloc_scratch_ptr(dev);
  if (scratch == nullptr) return ATTN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The tickets must start at zero; clear them in stream order (no allocation).
  if (cudaMemsetAsync(static_cast<unsigned char*>(scratch) + plan.ticket_off, 0, plan.total - plan.ticket_off, s) !=
      cudaSuccess)
    return ATTN_ERR_CUDA;
  if (d == 64)
    return dispatch_decode_gc<64>(q, k_cache, v_cache, seqlens, o, lse, B, Hq, Hkv, Lmax, scale, scratch, plan, s,
                                  dev);
  return dispatch_decode_gc<128>(q, k_cache, v_cache, seqlens, o, lse, B, Hq, Hkv, Lmax, scale, scratch, plan, s,
                                 dev);
}
