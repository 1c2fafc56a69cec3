/*
 * duo_attn.h -- C ABI of a GB300 (sm_103a) library for mixed-head causal attention
 * in long-context serving: retrieval heads over a full KV cache, streaming heads
 * over a sink + ring-buffer cache.
 *
 * What the operations compute (sources are the pages this library restates):
 *
 *   DuoAttention README (mit-han-lab/duo-attention), Abstract: a few attention heads
 *   ("retrieval heads") need full attention over every token and keep a full KV
 *   cache; the others ("streaming heads") look mostly at the attention sinks and
 *   the recent tokens and keep a constant-size cache. With S = sink_size and
 *   R = recent_size (quick start: S = 64, R = 256), query position i of a head sees
 *   key position j when
 *       retrieval:  j <= i
 *       streaming:  j <= i  and  (j < S  or  i - j < R)
 *   and the output is softmax(q.k / sqrt(head_dim)) over the visible keys, times v.
 *
 *   vLLM issue "Could you support Attention Sink?", block tables and its option 3:
 *   sink tokens stay in their own slots and later tokens wrap around a circular
 *   buffer, so nothing is ever moved. Token t is stored in slot t if t < S, else in
 *   slot S + ((t - S) mod R).
 *
 *   transformers pull request "[WIP] Dynamic length in static cache": a decode step
 *   attends only to the positions written so far, never to the unused capacity.
 *
 * Conventions for every call:
 *   - All tensors are caller-owned device memory (e.g. torch tensors); the library
 *     allocates no device memory and never synchronises the device, except in
 *     duo_device_error().
 *   - bf16 means IEEE-754 binary16 "brain float" (torch.bfloat16). Tensors are dense
 *     and row-major in the index order written; base addresses must be 16-byte
 *     aligned.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Every kernel runs on it, asynchronously to the host. The append and decode
 *     kernels use programmatic dependent launch among themselves (an append lets the
 *     decode after it start early, each waits for the grid before it before touching
 *     its data); stream order holds as usual for any kernel launched without the
 *     cudaLaunchAttributeProgrammaticStreamSerialization attribute. A caller kernel
 *     launched with that attribute right after an append or a decode must call
 *     cudaGridDependencySynchronize() before it reads what they wrote.
 *   - Arguments are checked on the host before any launch. On an error nothing is
 *     written, the cache length is unchanged, the status is returned and
 *     duo_last_error() describes it.
 *   - A handle holds host state only; it may be used from one host thread at a
 *     time. The device is the one current when duo_create ran.
 */
#ifndef DUO_ATTN_H_
#define DUO_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DUO_OK = 0,
  DUO_ERR_INVALID_ARG = 1,    /* null pointer, bad size, misaligned address */
  DUO_ERR_UNSUPPORTED = 2,    /* a shape the kernels do not implement (see duo_config) */
  DUO_ERR_CAPACITY = 3,       /* the append would exceed max_seq_len */
  DUO_ERR_CUDA = 4,           /* a CUDA runtime or driver call failed (launch error) */
  DUO_ERR_DEVICE_TIMEOUT = 5, /* a kernel gave up a bounded wait (see duo_device_error) */
  DUO_ERR_WORKSPACE = 6       /* decode workspace missing or smaller than required */
} duo_status;

/* Head kinds, one per KV head. A query head h uses KV head h / (num_q_heads /
 * num_kv_heads) and inherits its kind. */
#define DUO_STREAMING 0
#define DUO_RETRIEVAL 1

typedef struct {
  int32_t batch;        /* B >= 1 */
  int32_t num_q_heads;  /* Hq, a multiple of num_kv_heads, Hq / Hkv in {1, 2, 4, 8} */
  int32_t num_kv_heads; /* Hkv, 1 ... 128 */
  int32_t head_dim;     /* D in {64, 128} */
  int32_t sink_size;    /* S >= 0 */
  int32_t recent_size;  /* R >= 1 (R = 0 would leave a query with no key) */
  int64_t max_seq_len;  /* capacity of each retrieval head's cache, in tokens */
} duo_config;

typedef struct duo_handle duo_handle;

/* The caches of one layer. All pointers are device pointers owned by the caller.
 *   k_full, v_full : bf16 [B, n_ret, max_seq_len, D]; row t of retrieval head r holds
 *                    token t for t < n. Rows >= n are never read.
 *   k_sr, v_sr     : bf16 [B, n_str, S + R, D]; the sink slots then the ring slots of
 *                    each streaming head.
 *   pos            : int32 [B, S + R]; the token position held by each slot, -1 if
 *                    empty. Shared by all streaming heads of a sequence.
 *   n              : tokens appended so far (the same for every sequence of the batch).
 * n_ret / n_str are the numbers of retrieval / streaming KV heads; a pointer whose
 * count is zero may be NULL. The compact order of heads of one kind is increasing
 * KV-head index (see duo_classify_heads). Initialise a cache with duo_cache_reset. */
typedef struct {
  void* k_full;
  void* v_full;
  void* k_sr;
  void* v_sr;
  int32_t* pos;
  int64_t n;
} duo_kv_cache;

/* Per-head retrieval/streaming mask (host only, no device work).
 * is_retrieval[Hkv]: nonzero = retrieval. Writes kind_index[h] = the index of KV head
 * h among the heads of its kind (its plane in k_full/v_full or k_sr/v_sr), and
 * *n_retrieval. Source: the DuoAttention README's quick start turns trained per-head
 * gate values into a binary retrieval/streaming choice per head. */
duo_status duo_classify_heads(const uint8_t* is_retrieval, int32_t num_kv_heads, int32_t* kind_index,
                              int32_t* n_retrieval);

/* Create a handle for one layer shape and head mask (host arrays, copied). */
duo_status duo_create(const duo_config* config, const uint8_t* is_retrieval, duo_handle** out);
void duo_destroy(duo_handle* handle);

/* Re-classify the KV heads of an existing handle (host array of num_kv_heads flags,
 * copied), e.g. after loading another head pattern. The caches are laid out by kind
 * ([B, n_ret, ...] and [B, n_str, ...]), so the caller must re-lay them out (or reset
 * and refill them) for the new counts before the next call that uses them; the shape
 * of the handle is otherwise unchanged. The DuoAttention README's patch applies a
 * loaded head pattern the same way: one mask per layer. */
duo_status duo_set_head_mask(duo_handle* handle, const uint8_t* is_retrieval);

/* Empty the cache: pos[] := -1 on `stream`, cache->n := 0. */
duo_status duo_cache_reset(duo_handle* handle, duo_kv_cache* cache, void* stream);

/* Append T >= 1 new tokens at positions n ... n+T-1 and set cache->n += T.
 * k_new, v_new: bf16 [B, T, Hkv, D] (token-major, as a fused QKV projection emits).
 * Retrieval heads: rows n ... n+T-1 of k_full/v_full. Streaming heads: each token goes
 * to slot t (t < S) or S + ((t - S) mod R); of the tokens of one call only those still
 * held when the call ends are written (t < S, or t >= n+T-R), so the result equals T
 * single-token appends and no slot is written twice. pos[] is updated to match.
 * DUO_ERR_CAPACITY if n + T > max_seq_len (nothing written). */
duo_status duo_kv_append(duo_handle* handle, duo_kv_cache* cache, const void* k_new, const void* v_new, int32_t T,
                         void* stream);

/* Prefill attention of T >= 1 new tokens at positions n ... n+T-1 (n = cache->n, the
 * cache state BEFORE these tokens are appended; n = 0 for a one-shot prefill, n > 0
 * for a chunk of a chunked prefill against the growing cache).
 * q: bf16 [B, T, Hq, D]; k, v: bf16 [B, T, Hkv, D] of the same tokens; o: bf16
 * [B, T, Hq, D]. A retrieval head attends to cache rows [0, n) and to the new tokens;
 * a streaming head to what its sink + ring cache holds and to the new tokens, each
 * with the visibility rule above. Scale 1/sqrt(D) is applied in fp32 to the fp32
 * product; softmax and accumulation are fp32; o is rounded to nearest even.
 * The cache is not modified: call duo_kv_append(k, v) afterwards.
 * Fully masked key tiles are skipped, so a streaming head costs O((S + R) * T). */
duo_status duo_attn_prefill(duo_handle* handle, const duo_kv_cache* cache, const void* q, const void* k,
                            const void* v, int32_t T, void* o, void* stream);

/* As duo_attn_prefill, restricted to the query heads whose KV head kind bit is set in
 * kind_mask (bit 0 = streaming, bit 1 = retrieval). Rows of o for other heads are not
 * written. Used to time the retrieval heads alone. */
duo_status duo_attn_prefill_select(duo_handle* handle, const duo_kv_cache* cache, const void* q, const void* k,
                                   const void* v, int32_t T, void* o, int32_t kind_mask, void* stream);

/* Bytes of device workspace the decode entry points (duo_attn_decode, _paged, _varlen,
 * duo_dca_decode, duo_attn_decode_kv4) need for a cache of n tokens; the size covers
 * the largest grid any of them launches, so one workspace serves them all. */
size_t duo_decode_workspace_size(const duo_handle* handle, int64_t n);

/* One decode step for the token at position p = cache->n - 1, which must already have
 * been appended (duo_kv_append with T = 1). q: bf16 [B, Hq, D]; o: bf16 [B, Hq, D].
 * Reads rows [0, n) of each retrieval head and the valid slots of each streaming head
 * (each slot checked against pos[] and the visibility rule), every K/V byte once per
 * KV head for all its query heads. The keys are split over the GPU's SMs; partial
 * softmaxes (o, max, sum) go to `workspace` and are merged by log-sum-exp.
 * workspace: device memory of at least duo_decode_workspace_size(handle, n) bytes,
 * 256-byte aligned. It holds the partial softmax results (o, max, sum) of the
 * (sequence, KV head) pairs split over several CTAs, which a second kernel merges
 * right after the decode kernel (its programmatic dependent); nothing in it has to
 * survive between calls, so the memory may hold anything between calls.
 * Calls sharing one workspace must be ordered on the GPU (same stream). */
duo_status duo_attn_decode(duo_handle* handle, const duo_kv_cache* cache, const void* q, void* o, void* workspace,
                           size_t workspace_bytes, void* stream);

/* duo_attn_decode without a workspace argument, for callers that cannot allocate
 * device memory for scratch (an engine that has handed all device memory to its own
 * pool, a loop that must not call cudaMalloc/cudaFree because they may synchronise,
 * a runtime whose allocator owns every allocation). The pages have no counterpart:
 * it is an interface variant of the decode step above and computes the same result.
 * Scratch lives in a 2 MiB array inside the library (every GPU that loads the library
 * holds it until the process exits); shapes whose bf16 decode scratch (one partial
 * of g (D + 4) floats per CTA and per (sequence, KV head), with one CTA per SM)
 * exceeds 2 MiB get DUO_ERR_WORKSPACE. Nothing is
 * allocated: no cudaMalloc, cudaFree or allocating library call. The first call on
 * each device, and the first in any other CUDA context made current there later (after
 * cudaDeviceReset, say), looks up the array's device address (cudaGetSymbolAddress);
 * make that first call before any stream capture. All calls on a device share the
 * one array, so calls that overlap on the GPU (different streams, or several host
 * threads) race: order them on one stream. */
duo_status duo_attn_decode_static(duo_handle* handle, const duo_kv_cache* cache, const void* q, void* o,
                                  void* stream);

/* Paged caches, as a block allocator hands out memory in a serving engine (vLLM issue
 * "Could you support Attention Sink?" discusses the cache as fixed-size token blocks
 * chained by a block table, and keeping the first block as the sinks while dropping
 * the middle blocks and keeping the recent ones). With a duo_paged descriptor,
 * cache->k_full and cache->v_full are pools of blocks, bf16 [num_blocks, block_size,
 * D], shared by every sequence and head; row t of retrieval head r of sequence b is
 * row t % block_size of block block_table[(b * n_ret + r) * max_blocks + t / block_size].
 *
 * stream_table == NULL: streaming heads keep their sink + ring cache (cache->k_sr,
 * v_sr, pos). stream_table != NULL: streaming heads live in the same pools too, token
 * t of streaming head s of sequence b at row t % block_size of block
 * stream_table[(b * n_str + s) * max_blocks + t / block_size]; cache->k_sr, v_sr and pos
 * are then not used (may be NULL). Block granularity is only a storage choice: a query
 * still sees exactly the sinks and its recent window, token by token, so results match
 * the ring cache up to fp32 summation order. Once the cache holds n tokens, the blocks
 * duo_paged_stream_dead_blocks names hold no token any later query can see: the caller
 * may free them (their table entries are never read again). An append writes a
 * streaming token only if its block is still live when the call ends, so only live
 * blocks need to exist: the sink blocks and those reaching back R tokens from the end.
 *
 * The capacity of a head is block_size * max_blocks tokens (max_seq_len is not used).
 * A block id outside [0, num_blocks) that would be read or written is never
 * dereferenced: its rows are skipped and duo_device_error() reports
 * DUO_ERR_INVALID_ARG. Retrieval results equal the contiguous layout's, bit for bit. */
typedef struct {
  const int32_t* block_table;  /* int32 [B, n_ret, max_blocks], device memory (NULL if n_ret = 0) */
  int32_t block_size;          /* rows per block, a positive multiple of 128 */
  int32_t max_blocks;          /* table entries per (sequence, head) */
  int64_t num_blocks;          /* blocks in each pool */
  const int32_t* stream_table; /* int32 [B, n_str, max_blocks], device memory, or NULL */
} duo_paged;

/* Logical blocks [*lo, *hi) of a paged streaming head that no query at a position
 * >= n - 1 can see once the cache holds n tokens: blocks past the sink blocks
 * (lo = ceil(S / block_size)) that end at or before the recent window of the last
 * token (hi = max(lo, floor(max(0, n - R) / block_size))). The range only grows with
 * n, so after each call the caller may free [previous hi, hi). Host only. */
duo_status duo_paged_stream_dead_blocks(int32_t sink_size, int32_t recent_size, int32_t block_size, int64_t n,
                                        int64_t* lo, int64_t* hi);

duo_status duo_kv_append_paged(duo_handle* handle, duo_kv_cache* cache, const duo_paged* paged, const void* k_new,
                               const void* v_new, int32_t T, void* stream);
duo_status duo_attn_prefill_paged(duo_handle* handle, const duo_kv_cache* cache, const duo_paged* paged,
                                  const void* q, const void* k, const void* v, int32_t T, void* o, void* stream);
duo_status duo_attn_decode_paged(duo_handle* handle, const duo_kv_cache* cache, const duo_paged* paged,
                                 const void* q, void* o, void* workspace, size_t workspace_bytes, void* stream);

/* 4-bit KV caches. The DuoAttention README pairs the method with a 4-bit KV cache to
 * decode millions of tokens on one GPU (quick-start demo, Efficiency section) but gives
 * no format; this library uses the plainest asymmetric one. Each cached row (the D
 * values of one token of one head) is stored as D 4-bit codes plus an fp16 scale and
 * zero: scale = fp16((max - min) / 15), zero = fp16(min), code = clamp(rint((x - zero)
 * / scale), 0, 15) with every step in fp32 round-to-nearest (all codes 0 when the
 * scale is 0), value = code * scale + zero. Codes are packed two per byte, the even
 * dim in the low nibble. Rows must stay within the fp16 range.
 *
 * K codes are stored row by row (D / 2 bytes per row). V codes are stored in groups of
 * 16 rows (rows 16 m ... 16 m + 15 of a plane, 8 D bytes), ordered for the decode's
 * tensor-core fragments: the byte with the codes of dims 2 dp (low nibble) and 2 dp + 1
 * (high nibble) of row k of the group sits at byte
 *     4 ((4 (dp / MT) + (k % 8) / 2) MT + dp % MT) + 2 (k % 2) + k / 8,   MT = D / 16,
 * of the group. Each byte belongs to one row, so appending a row writes only its bytes.
 *
 * Layout (all device memory, caller-owned, 16-byte aligned), with cap16 = max_seq_len
 * and sr16 = S + R each rounded up to a multiple of 16 rows:
 *   k_codes, v_codes    u8  [B, n_ret, cap16, D / 2]   retrieval heads, row t = token t
 *   k_sz, v_sz          u32 [B, n_ret, cap16]          fp16 scale (low half), zero (high)
 *   ks_codes, vs_codes  u8  [B, n_str, sr16, D / 2]    streaming heads, sink + ring slots
 *   ks_sz, vs_sz        u32 [B, n_str, sr16]
 * cache->n and cache->pos keep their meaning; cache->k_full, v_full, k_sr, v_sr are not
 * used. duo_kv_append_kv4 quantizes and stores the new tokens (same slot rule as
 * duo_kv_append); duo_attn_decode_kv4 is duo_attn_decode over these arrays, with the
 * dequantization folded into the dot products (q . k = scale (q . codes) + zero sum(q)).
 * duo_attn_prefill_kv4 prefills a chunk against caches in this form.
 *
 * duo_attn_decode_kv4 runs its dot products on the tensor cores with fp16 operands
 * (codes, q, and p times the row scale, stored as p scale / 64) and fp32 accumulation,
 * so q must lie within the fp16 range as well (bf16 values there convert exactly).
 * Its workspace is the one duo_decode_workspace_size gives; it launches two CTAs per
 * SM. Errors: as duo_attn_decode, plus DUO_ERR_INVALID_ARG for a NULL or misaligned
 * array the handle's head kinds need (every array 16-byte aligned). */
typedef struct {
  void* k_codes;
  void* v_codes;
  void* k_sz;
  void* v_sz;
  void* ks_codes;
  void* vs_codes;
  void* ks_sz;
  void* vs_sz;
} duo_kv4_cache;

duo_status duo_kv_append_kv4(duo_handle* handle, duo_kv_cache* cache, const duo_kv4_cache* kv4, const void* k_new,
                             const void* v_new, int32_t T, void* stream);
duo_status duo_attn_decode_kv4(duo_handle* handle, const duo_kv_cache* cache, const duo_kv4_cache* kv4,
                               const void* q, void* o, void* workspace, size_t workspace_bytes, void* stream);

/* Prefill of T new tokens against 4-bit caches (chunked prefill after earlier chunks were
 * appended with duo_kv_append_kv4): as duo_attn_prefill, with the keys and values of the
 * cache rows (retrieval rows [0, n), valid sink + ring slots) read from `kv4` and
 * dequantized (code * scale + zero in fp32, rounded to bf16) into the kernel's shared-memory
 * tiles, so no bf16 copy of the cache exists anywhere; the T new tokens' k and v are the bf16
 * inputs as usual. Append the chunk afterwards with duo_kv_append_kv4. cache->k_full,
 * v_full, k_sr, v_sr are not used. Errors: as duo_attn_prefill, plus those of the 4-bit
 * arrays (see duo_attn_decode_kv4). */
duo_status duo_attn_prefill_kv4(duo_handle* handle, const duo_kv_cache* cache, const duo_kv4_cache* kv4,
                                const void* q, const void* k, const void* v, int32_t T, void* o, void* stream);

/* 4-bit caches with the retrieval rows in a paged pool (the two layouts above combined:
 * the block allocator of the attention-sink issue holding the 4-bit rows the README
 * pairs the method with). kv4->k_codes, v_codes are pools u8 [num_blocks, block_size,
 * D / 2] and kv4->k_sz, v_sz pools u32 [num_blocks, block_size]; row t of retrieval head
 * r of sequence b is row t % block_size of block paged->block_table[(b n_ret + r)
 * max_blocks + t / block_size] (block_size a multiple of 128, so 16-row V groups never
 * straddle blocks). The row encoding and the V group order are those of the contiguous
 * 4-bit arrays. Streaming heads keep their 4-bit sink + ring arrays: paged->stream_table
 * must be NULL (DUO_ERR_UNSUPPORTED otherwise). Capacity, bad block ids and errors: as
 * duo_kv_append_paged / duo_attn_decode_paged (a bad id is reported by duo_device_error,
 * its rows are neither written nor read). */
duo_status duo_kv_append_kv4_paged(duo_handle* handle, duo_kv_cache* cache, const duo_paged* paged,
                                   const duo_kv4_cache* kv4, const void* k_new, const void* v_new, int32_t T,
                                   void* stream);
duo_status duo_attn_decode_kv4_paged(duo_handle* handle, const duo_kv_cache* cache, const duo_paged* paged,
                                     const duo_kv4_cache* kv4, const void* q, void* o, void* workspace,
                                     size_t workspace_bytes, void* stream);

/* Dual Chunk Attention (vLLM pull request "[Model] Implement DualChunkAttention for
 * Qwen2 Models"): the sequence is cut into chunks of chunk_len positions from the start
 * (the last one may be shorter) and every position carries three query vectors made by
 * the rotary layer. Query i attends causally to every key j <= i with
 *     weight = (q_x(i) . k_j) * softmax_scale * mscale[i],   softmax_scale = 1/sqrt(D),
 * where q_x is q when j lies in i's chunk, q_succ when j lies in the chunk just before,
 * and q_inter for any earlier chunk; mscale is an fp32 per-position factor applied to
 * the fp32 product (NULL: 1). The pull request asks for this as one fused kernel in
 * place of three attention calls per chunk merged by log-sum-exp.
 *
 * Both entry points treat every head as full attention: the handle must have no
 * streaming head (DUO_ERR_UNSUPPORTED otherwise). chunk_len must be a positive multiple
 * of 256 (DUO_ERR_UNSUPPORTED otherwise) so that chunk boundaries fall on the
 * kernels' 256-row query blocks and 128-key tiles.
 *
 * duo_dca_prefill: prefill of T tokens at positions n ... n+T-1 against the cache as it
 * is before them (cache NULL or cache->n = 0: one-shot; else a chunk of a chunked
 * prefill, cache->n a multiple of 256, keys of rows [0, n) read from cache->k_full /
 * v_full). q, q_succ, q_inter: bf16 [B, T, Hq, D]; k, v: bf16 [B, T, Hkv, D]; mscale:
 * fp32 [B, T] (the chunk's positions) device memory or NULL; o: bf16 [B, T, Hq, D];
 * all device, 16-byte aligned. Append k and v with duo_kv_append afterwards. */
duo_status duo_dca_prefill(duo_handle* handle, const duo_kv_cache* cache, const void* q, const void* q_succ,
                           const void* q_inter, const void* k, const void* v, const float* mscale, int32_t T,
                           int32_t chunk_len, void* o, void* stream);

/* duo_dca_decode: one decode step at position cache->n - 1 (the token appended first)
 * over the retrieval caches. q, q_succ, q_inter: bf16 [B, Hq, D]; mscale: fp32 [B] or
 * NULL; o: bf16 [B, Hq, D]; workspace as for duo_attn_decode. */
duo_status duo_dca_decode(duo_handle* handle, const duo_kv_cache* cache, const void* q, const void* q_succ,
                          const void* q_inter, const float* mscale, int32_t chunk_len, void* o, void* workspace,
                          size_t workspace_bytes, void* stream);

/* Per-sequence lengths on the device: serving batches
 * hold sequences of different lengths, and a decode step whose lengths live in device
 * memory can be captured once in a CUDA graph and replayed step after step. The
 * transformers pull request "[WIP] Dynamic length in static cache" debates exactly
 * this: a length the compiled step reads at run time instead of a host integer.
 *
 * duo_kv_append_varlen: appends ONE token to every sequence b at position
 * seq_lens[b] (int32 [B], device memory, read and then advanced by one on the device).
 * k_new, v_new: bf16 [B, 1, Hkv, D]. Same slot rule as duo_kv_append. A sequence whose
 * retrieval cache is full is left unchanged and duo_device_error() reports
 * DUO_ERR_CAPACITY. cache->n is not used or changed. */
duo_status duo_kv_append_varlen(duo_handle* handle, duo_kv_cache* cache, int32_t* seq_lens, const void* k_new,
                                const void* v_new, void* stream);

/* duo_attn_decode with per-sequence lengths: sequence b holds seq_lens[b] tokens
 * (device int32 [B], values clamped to [0, max_len]) and its query is at position
 * seq_lens[b] - 1. The work split is planned for max_len (host, 1 ... max_seq_len),
 * so the launch shape does not depend on the device values; a sequence of length 0
 * gets a zero output. cache->n is not used. Workspace as for duo_attn_decode. */
duo_status duo_attn_decode_varlen(duo_handle* handle, const duo_kv_cache* cache, const int32_t* seq_lens,
                                  int64_t max_len, const void* q, void* o, void* workspace, size_t workspace_bytes,
                                  void* stream);

/* Synchronises the device, then returns (and clears) the OR of the error codes that
 * kernels of this library recorded when a bounded wait ran out, or when a device-side
 * append met a full cache; 0 = none. Sets *code and returns DUO_ERR_DEVICE_TIMEOUT if
 * a wait ran out, DUO_ERR_CAPACITY if the only error is a full cache. */
duo_status duo_device_error(uint32_t* code);

/* Self-test of failure detection (the pages have no counterpart): launches one
 * CTA that waits on an mbarrier nothing completes, with the same bounded wait
 * the attention kernels use but a limit of limit_us microseconds (1 ... 10^6).
 * The wait gives up and records an error code; a following duo_device_error()
 * returns DUO_ERR_DEVICE_TIMEOUT, and the CUDA context stays usable. */
duo_status duo_selftest_bounded_wait(uint32_t limit_us, void* stream);

/* Message describing the last error of the calling host thread ("" if none). */
const char* duo_last_error(void);

/* Short name of a status code. */
const char* duo_status_string(duo_status status);

#ifdef __cplusplus
}
#endif

#endif /* DUO_ATTN_H_ */
