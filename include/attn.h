/*
 * exact attention for sm_103a (B300): C ABI.
 *
 * Computes exact multi-head scaled-dot-product attention
 *     O = softmax(scale * Q K^T + causal mask) V
 * tile by tile with the blockwise (online) softmax recurrence, so the score
 * matrix never reaches device memory, plus the KV-cache decode form, with
 * MHA / GQA / MQA head sharing. Sources, cited by page title and section:
 *
 *   [MG-A] menggq.pages.dev, "Transformer 架构的数学与计算深度解析：注意力机制的
 *          详尽研究报告": §2.2 scores, §2.3 scaling, §2.4 softmax and weighted
 *          sum, §4.1 causal mask, §4.2 cross-attention, §6.3 online softmax.
 *   [AUT]  auturnal.com, "从注意力到 IO 感知执行：Transformer 的计算结构、复杂度
 *          与可复核分析" (v10): §4/§6 score bytes, §8 (m, l, u recurrence,
 *          first two equations), §9 (KV cache size, third equation).
 *   [IMR]  imreese.github.io, "Transformer 笔记：注意力机制为什么会变成系统问题":
 *          masking section, prefill/decode section.
 *   [PW]   pwwt.cn news 6124947: §2.1 S = QK^T / sqrt(d_k), §2.3 MQA/GQA,
 *          §3.1-3.2 KV cache, §4.2 tiling + online softmax is exact.
 *
 * Conventions for every entry point:
 *   - Tensors are bf16 (IEEE bfloat16 bit patterns), contiguous, row-major.
 *     Device pointers must be 16-byte aligned (LSE pointers 4-byte aligned).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). All work is asynchronous on that stream; no entry point
 *     synchronises except attn_device_status().
 *   - The caller owns every buffer, including the decode workspace. Nothing
 *     here allocates or frees device memory.
 *   - Argument errors are detected on the host and returned before anything
 *     is launched. Launch failures return ATTN_ERR_CUDA. Problems only the
 *     device can see (a bounded internal wait that gave up, a sequence length
 *     outside [0, Lmax]) are OR-ed into a per-device status word that
 *     attn_device_status() reads and clears.
 *   - GQA mapping: Hq % Hkv == 0 and query head h reads K/V head
 *     h / (Hq / Hkv) (contiguous groups; [PW] §2.3). Hkv == Hq is MHA,
 *     Hkv == 1 is MQA.
 *   - Head dimension d (= d_k = d_v) must be 64 or 128; anything else returns
 *     ATTN_ERR_UNSUPPORTED.
 */
#ifndef EXACT_ATTN_SM103_H
#define EXACT_ATTN_SM103_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1, /* bad pointer, size, alignment or scale */
  ATTN_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. d not in {64, 128}) */
  ATTN_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed */
  ATTN_ERR_TIMEOUT = 4,     /* (device) an internal pipeline wait gave up */
  ATTN_ERR_DEVICE_ARG = 5   /* (device) a decode length outside [0, Lmax] or a page id outside [0, num_pages) */
} attn_status;

/*
 * Prefill / cross-attention forward ([MG-A] §2.2-§2.4, §4.1-§4.2, §6.3;
 * [AUT] §8; [PW] §2.1, §4.2).
 *
 *   q   [B, Hq,  Nq, d] bf16 (device)    k, v [B, Hkv, Nk, d] bf16 (device)
 *   o   [B, Hq,  Nq, d] bf16 (device, written)
 *   lse [B, Hq,  Nq] fp32 (device, written) or NULL: natural log of the sum of
 *       exp(scale * q_i . k_j) over the keys row i sees; -inf for a row that
 *       sees no key (its o row is 0).
 *   scale: multiplies every score before the mask; must be finite and > 0
 *       (1/sqrt(d) gives the pages' scaled dot product, [MG-A] §2.3).
 *   causal: 0 = every query sees every key. 1 = query i sees key j iff
 *       j <= i + (Nk - Nq), i.e. the last query is aligned with the last key;
 *       for Nq == Nk this is the pages' rule j <= i ([IMR] masking section).
 *   Sizes: B, Hq, Hkv >= 1; Nq, Nk >= 0 (Nq == 0 is a no-op; Nk == 0 gives
 *       o = 0, lse = -inf, and k / v may then be NULL); ceil(Nq / 256) <=
 *       65535; B <= 65535.
 */
ATTN_API attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                     int Nq, int Nk, int d, float scale, int causal, void* stream);

/*
 * attn_fwd with a local (sliding) window ([AUT] §2, its Longformer
 * comparison: local windows change which positions interact; [PW] §6.1:
 * window attention costs O(n w)). Query i is aligned with key
 * i + (Nk - Nq) and sees key j only if |j - (i + Nk - Nq)| < window; with
 * causal = 1 also only j <= i + (Nk - Nq). window = 0 is no window (attn_fwd);
 * window < 0 is ATTN_ERR_INVALID_ARG. Rows that see no key give o = 0,
 * lse = -inf. Only the key tiles a query tile can see are read. Other
 * arguments as attn_fwd.
 */
ATTN_API attn_status attn_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                                     int Hkv, int Nq, int Nk, int d, float scale, int causal, int window,
                                     void* stream);

/*
 * attn_fwd on tensors that live in host memory. The same operation and
 * arguments as attn_fwd ([MG-A] §2.2-§2.4, §4.1), except that q, k, v, o and
 * lse are HOST pointers (page-locked memory lets the copies overlap; pageable
 * memory works but the copies then serialise).
 *
 * Work moves in chunks: the K and V of one (batch, KV head) group go to the
 * device once, then its query heads in chunks of a few heads each (as many as
 * fill about two CTAs per SM): a chunk's Q goes in, the prefill runs on it,
 * its O and LSE come back. Chunks are pipelined through ATTN_FWD_HOST_SLOTS
 * staging slots (and K, V through two) of the caller's device workspace, so
 * the copy in of one chunk, the prefill of the one before and the copy out of
 * the one before that run at the same time (two copy streams of the library
 * beside `stream`, which runs the prefill kernels). The result is bit for bit
 * that of attn_fwd. The call returns once everything is queued; when `stream`
 * has reached the point of the call, o and lse are complete in host memory.
 *
 *   workspace / workspace_bytes: device memory of at least
 *       attn_fwd_host_workspace_size(B, Hq, Hkv, Nq, Nk, d) bytes, 256-byte
 *       aligned, not touched by anything else until `stream` passes the call.
 *   The first call on a device creates the two copy streams and the events
 *   it synchronises with (kept until the process exits). Calls on one device
 *   are serialised on the host while they queue their work.
 *   q and o may be NULL when Nq == 0, k and v when Nk == 0.
 *   Returns the errors of attn_fwd, plus ATTN_ERR_INVALID_ARG for a missing
 *   or too small workspace.
 */
#define ATTN_FWD_HOST_SLOTS 3
ATTN_API size_t attn_fwd_host_workspace_size(int B, int Hq, int Hkv, int Nq, int Nk, int d);
ATTN_API attn_status attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                                   int Hkv, int Nq, int Nk, int d, float scale, int causal, void* workspace,
                                   size_t workspace_bytes, void* stream);

/*
 * Workspace bytes attn_fwd_rope needs: the rotated K ([B, Hkv, Nk, d] bf16)
 * and two layouts (position-major, pair-major) of a (cos, sin) table of
 * max(Nk, Nq) positions x d/2 pairs (fp32).
 * 0 for arguments attn_fwd_rope would reject.
 */
ATTN_API size_t attn_fwd_rope_workspace_size(int B, int Hkv, int Nq, int Nk, int d);

/*
 * attn_fwd_window with rotary position embedding applied to Q and K first
 * ([PW] §5.3): the components of each vector are split into pairs (2i, 2i+1)
 * and the pair of a vector at position m is rotated by m * base^(-2i/d), so
 * that scores depend only on relative position. Key j sits at position j and
 * query i at position i + (Nk - Nq). The rotated Q and K are rounded to bf16.
 * K is rotated once into the workspace (two small kernels: the (cos, sin)
 * table, then K); each Q tile is rotated inside the prefill kernel right
 * after it is loaded. q and k are not modified.
 *
 *   rope_base  > 1 and finite (10000 in the pages).
 *   workspace  >= attn_fwd_rope_workspace_size(B, Hkv, Nq, Nk, d) bytes,
 *              256-byte aligned, contents irrelevant (overwritten).
 * Other arguments as attn_fwd_window (Nk must be >= 1).
 */
ATTN_API attn_status attn_fwd_rope(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                                   int Hkv, int Nq, int Nk, int d, float scale, int causal, int window,
                                   float rope_base, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Workspace bytes attn_bwd needs: 72 bytes per query row (two fp32 values and
 * two 32-byte operand rows), each head's rows padded to a multiple of 128.
 * 0 for arguments attn_bwd would reject.
 */
ATTN_API size_t attn_bwd_workspace_size(int B, int Hq, int Nq);

/*
 * Backward pass of attn_fwd (causal or not, MHA/GQA/MQA): given the forward's
 * inputs, its output o and row LSE, and dout = dL/dO, writes dq = dL/dQ,
 * dk = dL/dK and dv = dL/dV. The scores are recomputed from q, k and lse
 * instead of being stored ([MG-A] §3.3; [MG-B] §3.2): with P = softmax(scale
 * Q K^T + mask), dV = P^T dO, dS = P * (dO V^T - rowsum(dO * O)),
 * dQ = scale dS K, dK = scale dS^T Q; the query heads of a GQA group add
 * into their shared dK, dV. No atomics: the result is deterministic.
 *
 *   q, dout, o  [B, Hq, Nq, d] bf16 (device); o as written by attn_fwd
 *   k, v        [B, Hkv, Nk, d] bf16 (device)
 *   lse         [B, Hq, Nq] fp32 (device), natural log, as written by
 *               attn_fwd (-inf for a row that sees no key); required
 *   dq          [B, Hq, Nq, d] bf16 (device, written)
 *   dk, dv      [B, Hkv, Nk, d] bf16 (device, written)
 *   workspace   >= attn_bwd_workspace_size(B, Hq, Nq) bytes, 256-byte
 *               aligned, contents irrelevant (overwritten)
 * Rows of dq that see no key are 0; keys no query sees get dk = dv = 0.
 * scale, causal (bottom-right aligned when Nq != Nk), d and the alignment
 * rules as attn_fwd; ceil(Nq / 128), B and Hkv <= 65535, else
 * ATTN_ERR_UNSUPPORTED. Three kernels: a per-row prologue on `stream`, then
 * dK/dV on `stream` and dQ beside it on a library stream of lower priority
 * (created once per device). `stream` waits for dQ through an event, so work
 * queued on `stream` after the call sees all three gradients, as if every
 * kernel had run on it. Calls from several host threads enqueue one at a
 * time.
 */
ATTN_API attn_status attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                              const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Nq, int Nk,
                              int d, float scale, int causal, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Size in bytes of the device workspace attn_decode needs for these sizes
 * (split-KV partial results and one ticket per (sequence, KV head, query
 * group)). Returns 0 for arguments attn_decode would reject. The workspace
 * must be zero-filled before its first use; every call that completes
 * leaves it zero-filled again, so it can be reused across calls on one
 * stream (calls that overlap on the device must use separate workspaces).
 * A call after which attn_device_status() reports ATTN_ERR_TIMEOUT can leave
 * part-counted tickets behind: zero-fill the workspace again before reusing it.
 */
ATTN_API size_t attn_decode_workspace_size(int B, int Hq, int Hkv, int Lmax, int d);

/*
 * KV-cache decode: one new query token per sequence attends to its cached
 * keys/values 0 .. seqlens[b]-1 ([IMR] prefill/decode section; [PW] §3.1-§3.2).
 * The caller has already appended the new token's K/V to the cache.
 *
 *   q        [B, Hq, d] bf16 (device)
 *   k_cache, v_cache [B, Hkv, Lmax, d] bf16 (device); rows at or past
 *            seqlens[b] are never used in the result.
 *   seqlens  [B] int32 (device), each in [0, Lmax]. A length of 0 gives
 *            o = 0, lse = -inf. A value outside the range is clamped into it
 *            and flagged in the device status (ATTN_ERR_DEVICE_ARG).
 *   o        [B, Hq, d] bf16 (device, written)
 *   lse      [B, Hq] fp32 (device, written) or NULL (natural log, as attn_fwd)
 *   workspace / workspace_bytes: device buffer of at least
 *            attn_decode_workspace_size(B, Hq, Hkv, Lmax, d) bytes, 16-byte
 *            aligned, zero-filled before first use (see above).
 */
ATTN_API attn_status attn_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* seqlens, void* o,
                        float* lse, int B, int Hq, int Hkv, int Lmax, int d, float scale, void* workspace,
                        size_t workspace_bytes, void* stream);

/*
 * Workspace bytes attn_decode_paged needs (0 for arguments it would reject).
 * Same rules as attn_decode_workspace_size, with Lmax = max_pages_per_seq *
 * page_size.
 */
ATTN_API size_t attn_decode_paged_workspace_size(int B, int Hq, int Hkv, int max_pages_per_seq, int page_size, int d);

/*
 * KV-cache decode over a paged cache, with the new token's K/V appended first.
 *
 * The cache is cut into fixed-size pages that are allocated on demand and need
 * not be contiguous; a per-sequence block table maps logical page numbers to
 * physical pages ([IMR] section "FlashAttention 和 PagedAttention 不是同一种
 * 答案"; [PW] §3.3). The new token joins the cache before the query attends
 * to it ([PW] §3.1).
 *
 *   q            [B, Hq, d] bf16 (device)
 *   k_new, v_new [B, Hkv, d] bf16 (device), or both NULL (no append)
 *   k_pages, v_pages [num_pages, Hkv, page_size, d] bf16 (device). Position p
 *                of sequence b is row p % page_size of physical page
 *                block_table[b * max_pages_per_seq + p / page_size].
 *   block_table  [B, max_pages_per_seq] int32 (device); entries past a
 *                sequence's last page are never read. An id outside
 *                [0, num_pages) is flagged in the device status
 *                (ATTN_ERR_DEVICE_ARG) and read as page 0.
 *   seqlens      [B] int32 (device): tokens already cached. With an append the
 *                new K/V is written at position seqlens[b] (the caller must
 *                have mapped that position to a page) and the query attends to
 *                positions 0..seqlens[b]; without one, to 0..seqlens[b]-1.
 *                Lengths outside [0, capacity - (append ? 1 : 0)], capacity =
 *                max_pages_per_seq * page_size, are clamped and flagged.
 *   o, lse       as attn_decode.
 *   page_size    a divisor of 128 that is >= 8, or a multiple of 128
 *                (others: ATTN_ERR_UNSUPPORTED).
 *   workspace    >= attn_decode_paged_workspace_size(...) bytes, zero-filled
 *                before first use, left zero-filled by every completed call
 *                (zero-fill it again after a call that timed out, as for
 *                attn_decode).
 * The appended rows are the only cache memory written.
 */
ATTN_API attn_status attn_decode_paged(const void* q, const void* k_new, const void* v_new, void* k_pages,
                                       void* v_pages, const int32_t* block_table, const int32_t* seqlens, void* o,
                                       float* lse, int B, int Hq, int Hkv, int num_pages, int page_size,
                                       int max_pages_per_seq, int d, float scale, void* workspace,
                                       size_t workspace_bytes, void* stream);

/*
 * Synchronises `stream`, then reads and clears the calling thread's current
 * device's status word. Returns ATTN_OK, ATTN_ERR_TIMEOUT or
 * ATTN_ERR_DEVICE_ARG (timeout wins if both are set), or ATTN_ERR_CUDA if
 * the synchronisation itself failed. If `detail` is not NULL it receives the
 * raw words {flags, wait site, block index}.
 */
ATTN_API attn_status attn_device_status(void* stream, unsigned* detail);

/* Human-readable name of a status code (static string, never NULL). */
ATTN_API const char* attn_status_string(attn_status s);

/* Bytes of an explicitly stored score matrix: heads * n^2 * bytes_per_score
 * ([AUT] §4 and §6: 512/1024/2048/4096 -> 1/4/16/64 MiB per fp32 head). */
ATTN_API uint64_t attn_score_bytes(int64_t n, int64_t heads, int bytes_per_score);

/* KV cache bytes 2 * layers * n * h_kv * d_h * bytes ([AUT] §9, third
 * equation; [PW] §3.2). */
ATTN_API uint64_t attn_kv_cache_bytes(int64_t layers, int64_t n, int64_t h_kv, int64_t d_h, int bytes_per_scalar);

/*
 * Decode without any caller-provided or library-allocated device memory.
 *
 * The paper has no counterpart for this entry point; it exists for callers
 * that cannot call cudaMalloc or hand over a workspace: for example code
 * running where allocation is forbidden or unsafe (inside a custom allocator
 * or memory-pool callback, under a framework that owns all device memory, or
 * at a point where an allocation could trigger a synchronising garbage
 * collection or fail under memory pressure).
 *
 * It computes exactly what attn_decode computes (same arguments, minus the
 * workspace), but the split-KV scratch lives in one static device array of
 * ATTN_NOALLOC_SCRATCH_BYTES bytes inside this library. Every GPU that loads
 * the library holds that array until the process exits.
 *
 *   - The caller still passes q, the caches, seqlens, o and (optionally) lse.
 *   - Returns ATTN_ERR_UNSUPPORTED when the problem would need more scratch
 *     than the array holds, i.e. when
 *     attn_decode_workspace_size(B, Hq, Hkv, Lmax, d) > ATTN_NOALLOC_SCRATCH_BYTES.
 *   - The first call on each device looks up the array's device address
 *     (with that device current); make that first call before any stream
 *     capture.
 *   - All calls share the one array, and it keeps the last call's contents:
 *     each call first clears the part that must start at zero, on `stream`.
 *     Calls whose work overlaps on the GPU (different streams, or different
 *     host threads on the same device) race on the array and must be
 *     serialised by the caller.
 *   - Nothing is allocated or freed: no cudaMalloc, no cudaFree, no library
 *     routine that allocates.
 */
#define ATTN_NOALLOC_SCRATCH_BYTES (8u << 20) /* 8 MiB */
ATTN_API attn_status attn_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                         const int32_t* seqlens, void* o, float* lse, int B, int Hq, int Hkv,
                                         int Lmax, int d, float scale, void* stream);

/*
 * Test hook for failure detection. The pages have no counterpart: it exists so
 * that the kernels' give-up path can be exercised on a GPU without a fault or
 * a hang.
 *
 * Every internal wait of the kernels is bounded (1 s). When one gives up, the
 * kernel records ATTN_ERR_TIMEOUT and, for the first wait of the launch to give
 * up, its site and block in the status word. The other roles of that CTA stop
 * waiting: at once in the prefill and decode, and in the backward at their own
 * limit (its elementwise and copy waits do not watch for an abort, which keeps
 * their polling light). The copies and MMAs still in flight are allowed to
 * land, tensor memory is freed and the kernel returns; attn_device_status()
 * then reports it.
 *
 * attn_test_arm_stall(kind) arms the next launch, in this process, of one
 * kernel: in its first CTA one role waits on a barrier that nothing ever
 * arrives on, with a 1 ms limit, instead of its first real wait:
 *   ATTN_TEST_STALL_PREFILL  attn_fwd / _window / _rope: the softmax warps of
 *                            query tile 0, first score tile (wait site 8)
 *   ATTN_TEST_STALL_DECODE   attn_decode / _paged / _noalloc: warp 0, first
 *                            K/V tile (wait site 20)
 *   ATTN_TEST_STALL_BACKWARD attn_bwd (a call with queries and keys): the dK/dV
 *                            kernel's elementwise warps of query columns
 *                            0-63, first score tile (wait site 38)
 * The hook disarms itself at that launch; kind 0 disarms it. The outputs of
 * the stalled launch are undefined, and a decode workspace it used must be
 * zero-filled again before reuse (its tickets are left part-counted). Returns
 * ATTN_ERR_INVALID_ARG for an unknown kind.
 */
#define ATTN_TEST_STALL_PREFILL 1
#define ATTN_TEST_STALL_DECODE 2
#define ATTN_TEST_STALL_BACKWARD 3
ATTN_API attn_status attn_test_arm_stall(int kind);

/* Library version string, e.g. "exact-attn-sm103 0.1". */
ATTN_API const char* attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* EXACT_ATTN_SM103_H */
