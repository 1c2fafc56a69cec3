// Internal types shared by the host API (duo_api.cu) and the kernel translation
// units. Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace duo {

// Upper bound of any single wait inside a kernel (an mbarrier phase). Normal
// waits last microseconds; running out means a bug, never a slow GPU.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

constexpr int kMaxHeads = 128;

// Error codes kernels OR into their error word.
enum : uint32_t {
  kErrPrefillProducer = 1u << 0,
  kErrPrefillMma = 1u << 1,
  kErrPrefillSoftmax = 1u << 2,
  kErrDecodeProducer = 1u << 8,
  kErrDecodeConsumer = 1u << 9,
  kErrSelftest = 1u << 16,
  kErrAppendCapacity = 1u << 20,
  kErrBadBlock = 1u << 21,
};

struct Shape {
  int B, Hq, Hkv, D, S, R, g, n_ret, n_str;
  int64_t cap;  // retrieval cache capacity (tokens)
};

// Compact head lists: KV head of the r-th retrieval / s-th streaming head, and
// for every KV head its kind and index within its kind.
struct HeadTable {
  uint8_t ret_head[kMaxHeads];
  uint8_t str_head[kMaxHeads];
  uint8_t kind[kMaxHeads];
  uint8_t kidx[kMaxHeads];
};

// Optional paged layout of the retrieval caches: k_full / v_full are pools of
// blocks [num_blocks, block_size, D]; row r of plane (b, ri) is row r % block_size
// of block table[(b * n_ret + ri) * max_blocks + r / block_size].
struct PagedLayout {
  const int32_t* table;  // nullptr = contiguous [B, n_ret, cap, D]
  int32_t block_size;    // a multiple of 128
  int32_t max_blocks;
  int64_t num_blocks;
  const int32_t* stream_table;  // streaming heads in the pool too (row = position); nullptr = ring caches
};

// Element offset in the pool of row r of plane `plane` of a block table; -1 if its
// block id is out of range.
__host__ __device__ __forceinline__ int64_t pool_row(const PagedLayout& pg, const int32_t* table, int D,
                                                     int64_t plane, int64_t r) {
  const int64_t blk = table[plane * pg.max_blocks + r / pg.block_size];
  if (blk < 0 || blk >= pg.num_blocks) return -1;
  return (blk * pg.block_size + r % pg.block_size) * D;
}

// Element offset of row r of retrieval plane `plane`; -1 if its block id is out of range.
__host__ __device__ __forceinline__ int64_t retrieval_row(const PagedLayout& pg, int64_t cap, int D, int64_t plane,
                                                          int64_t r) {
  if (!pg.table) return (plane * cap + r) * D;
  return pool_row(pg, pg.table, D, plane, r);
}

// ------------------------------------------------------------------ append
struct AppendParams {
  const uint16_t* k_new;  // bf16 [B, T, Hkv, D]
  const uint16_t* v_new;
  uint16_t* k_full;  // bf16 [B, n_ret, cap, D]
  uint16_t* v_full;
  uint16_t* k_sr;  // bf16 [B, n_str, S+R, D]
  uint16_t* v_sr;
  int32_t* pos;  // int32 [B, S+R]
  int64_t n;     // tokens before this call
  int T;
  // tokens of this call still held by a streaming head when it ends:
  // positions [sink_lo, sink_lo + sink_cnt) and [ring_lo, ring_lo + ring_cnt)
  int64_t sink_lo, sink_cnt, ring_lo, ring_cnt;
  Shape sh;
  HeadTable heads;
  PagedLayout pg;
  // 4-bit caches (k4 != nullptr), laid out as in DecodeParams
  uint8_t* k4;
  uint8_t* v4;
  uint8_t* ks4;
  uint8_t* vs4;
  uint32_t* ksz;
  uint32_t* vsz;
  uint32_t* kssz;
  uint32_t* vssz;
  int64_t cap16;
  int sr16;
};
cudaError_t launch_append(const AppendParams& p, int num_sms, cudaStream_t stream);
// 4-bit caches: quantizes and writes the rows the call keeps (same intervals).
cudaError_t launch_append_kv4(const AppendParams& p, int num_sms, cudaStream_t stream);
// One token per sequence at the position held in seq_lens[b] (device), which is
// then advanced; T is 1 and n is unused.
cudaError_t launch_append_varlen(const AppendParams& p, int32_t* seq_lens, cudaStream_t stream);
cudaError_t append_read_clear_error(uint32_t* code);

// ------------------------------------------------------------------ decode
constexpr int kDecodeTK = 128;  // keys per decode tile
constexpr int kDecodeTKKv4 = 256;  // keys per decode tile over 4-bit caches (32 per warp)
constexpr int kDecodeShortTiles = 4;  // caches of at most this many tiles: one CTA per unit
// CTAs per SM of the 4-bit decode (its rings are small enough for two; more warps hide
// the latency of its per-slice dependency chains); the bf16 decode runs one
constexpr int kDecodeCtasPerSmKv4 = 2;

struct DecodeParams {
  const uint16_t* q;  // bf16 [B, Hq, D]
  uint16_t* o;        // bf16 [B, Hq, D]
  const uint16_t* k_full;
  const uint16_t* v_full;
  const uint16_t* k_sr;
  const uint16_t* v_sr;
  const int32_t* pos;
  int64_t n;       // keys held by a retrieval head; the query is at position n - 1
  const int32_t* seq_lens;  // optional [B] device lengths (then n = the planned maximum)
  int nvalid;      // valid ring slots, min(n, S + R)
  int U_r, U_s;    // units (one per (sequence, KV head)) of each kind
  int64_t tiles_r; // key tiles per retrieval unit
  int64_t tiles_s; // key tiles per streaming unit
  int s_sink_tiles, s_win_lo;  // streaming heads in the pool: local tile lt reads row tile lt
                               // (lt < s_sink_tiles), else s_win_lo + lt - s_sink_tiles
  int64_t W;       // retrieval tiles: U_r * tiles_r
  int C;           // CTAs; CTA c < Cr takes retrieval tiles [c W / Cr, (c+1) W / Cr), and
                   // every CTA c streaming units c, c + C, ...
  int Cr;          // CTAs sharing the retrieval tiles: min(C, W), so none of them gets an
                   // empty share inside a unit's span (its partial would never arrive)
  int s_first;     // streaming units are dealt round-robin starting at this CTA
  float scale_log2;    // log2(e) / sqrt(D)
  float* partials;     // [C + U_r + U_s][g][D + 4] (o, max, sum, 2 pad) per segment
  Shape sh;
  HeadTable heads;
  PagedLayout pg;
  // Dual Chunk Attention (chunk_len > 0; every head full attention): the query vectors
  // for keys one chunk back and further back, and a per-sequence scale
  const uint16_t* q_succ;  // bf16 [B, Hq, D]
  const uint16_t* q_inter;
  const float* mscale;     // fp32 [B] or nullptr (1)
  int chunk_len;           // 0: not DCA; else a multiple of 256
  // 4-bit caches (k4 != nullptr): codes u8 [planes, pitch, D/2] and per-row fp16
  // (scale, zero) pairs u32 [planes, pitch]; pitch = cap16 for retrieval planes
  // (B * n_ret), sr16 for ring planes (B * n_str), both multiples of 16
  const uint8_t* k4;
  const uint8_t* v4;
  const uint8_t* ks4;
  const uint8_t* vs4;
  const uint32_t* ksz;
  const uint32_t* vsz;
  const uint32_t* kssz;
  const uint32_t* vssz;
  int64_t cap16;
  int sr16;
  int kv4;  // 4-bit caches (the retrieval arrays are null when there is no retrieval head)
};
size_t decode_workspace_bytes(const Shape& sh, int num_ctas);

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream);

// ------------------------------------------------------------------ prefill
constexpr int kPrefillBM = 128;        // query rows per query tile
constexpr int kPrefillBN = 128;        // keys per KV tile
constexpr int kPrefillRowsPerCta = 256;  // two query tiles per CTA

struct PrefillParams {
  CUtensorMap tm_q;      // 4-D over q [B, T, Hq, D], box 64 x 1 x 128 x 1, 128B swizzle
  CUtensorMap tm_k;      // 4-D over k [B, T, Hkv, D]
  CUtensorMap tm_v;      // 4-D over v [B, T, Hkv, D]
  CUtensorMap tm_kfull;  // 3-D over k_full [B * n_ret, n (extent), D]; paged: over the pool
  CUtensorMap tm_vfull;  //   [num_blocks, block_size, D]
  CUtensorMap tm_klast;  // paged only: the pool with row extent n % block_size (last block)
  CUtensorMap tm_vlast;
  CUtensorMap tm_ksr;    // 3-D over k_sr [B * n_str, nvalid (extent), D]
  CUtensorMap tm_vsr;
  uint16_t* o;           // bf16 [B, T, Hq, D]
  const int32_t* pos;    // int32 [B, S+R]
  int64_t n;             // cache length before the chunk (absolute position of row 0)
  int T;
  int nvalid;            // valid ring slots before the chunk
  int num_qt;            // 256-row query blocks per head: ceil(T / 256)
  int items_r;           // work items of retrieval heads: B * n_ret * g * num_qt
  int items_s;           // work items of streaming heads
  int qp_group;          // query blocks per group in the retrieval work order (>= 1)
  float scale_log2;
  Shape sh;
  HeadTable heads;
  PagedLayout pg;
  // Dual Chunk Attention (chunk_len > 0; every head full attention; cache length n a
  // multiple of 256): the query vectors for keys one chunk back and further back, and a
  // per-position scale
  CUtensorMap tm_qs;     // 4-D over q_succ [B, T, Hq, D], as tm_q
  CUtensorMap tm_qi;     // 4-D over q_inter [B, T, Hq, D]
  const float* mscale;   // fp32 [B, T] or nullptr (1)
  int chunk_len;         // 0: not DCA; else a multiple of 256
  // 4-bit caches (kv4 != 0): the cache tiles are dequantized into the K/V tiles in shared
  // memory instead of loaded by TMA; arrays laid out as in DecodeParams
  const uint8_t* k4;
  const uint8_t* v4;
  const uint8_t* ks4;
  const uint8_t* vs4;
  const uint32_t* ksz;
  const uint32_t* vsz;
  const uint32_t* kssz;
  const uint32_t* vssz;
  int64_t cap16;
  int sr16;
  int kv4;
};
cudaError_t launch_prefill(const PrefillParams& p, cudaStream_t stream);

// Error words of the kernel translation units (synchronous read-and-clear).
cudaError_t prefill_read_clear_error(uint32_t* code);
cudaError_t decode_read_clear_error(uint32_t* code);
cudaError_t selftest_read_clear_error(uint32_t* code);
cudaError_t launch_selftest_wait(uint64_t limit_ns, cudaStream_t stream);

}  // namespace duo
