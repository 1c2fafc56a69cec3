// duo_attn_decode: one query token per sequence against the caches, split over
// the GPU's SMs, merged by log-sum-exp.
//
// Work list. A "unit" is one (sequence, KV head): a retrieval unit holds n keys
// (rows [0, n) of its full cache), a streaming unit min(n, S + R) ring slots.
// Retrieval units are cut into tiles of kTK keys (256 over 4-bit caches) laid end
// to end; CTA c < Cr takes tiles [c W / Cr, (c + 1) W / Cr) with Cr = min(C, W), so
// no share is empty and
// every SM streams the same number of key bytes however long the contexts are
// (an empty share inside a unit's span would be counted as a part of the unit that
// never arrives). Streaming units (at most S + R keys) are
// dealt whole, round-robin: CTA c also takes units c, c + C, ... Only the n
// written positions are ever read, never the capacity (the transformers
// "Dynamic length in static cache" rule).
//
// Per CTA: eight warps; warp w owns keys [w kKPW, (w + 1) kKPW) of every tile and
// streams its own rows of K and V into a private 3-stage shared-memory ring with
// 1-D bulk copies (cp.async.bulk, completion on the warp's mbarrier). A warp
// refills a stage as soon as it has finished with it, so no producer warp and no
// cross-warp hand-off is needed, and each thread keeps up to 255 registers. The
// 4-bit decode gives each warp 32 keys of a 256-key tile, keeps 2 stages per warp and
// runs two CTAs per SM (128 registers).
//
// Inside a warp, LPK lanes share a key row and each owns 16 (or 8) of its dims:
// 128-bit shared loads, fp32 q pre-scaled by log2(e)/sqrt(D), packed fp32x2 FMAs
// for q.k of all g query heads of the KV head (every K and V byte is read once
// for all of them). The partial dot products are reduced across the lanes of a
// key by a reduce-scatter: at each of the first log2(g) shuffle steps a lane
// keeps half of its heads and sends the other half, so after log2(LPK) steps each
// lane holds the full score of one head (lane-dependent head order makes every
// step a plain add). The softmax then runs once per (key, head), the online
// state (running max with lazy rescaling: it moves only when a score exceeds it
// by 2^8, and running sum) is per lane for its head, and p of the other heads is
// fetched by shuffles for the packed p.v FMAs. With four or more query heads per KV
// head a warp's slice is instead two warp-level tensor-core MMAs (S = Q K^T, then
// O^T += V^T P^T; see MmaSlice), which takes the per-element FMAs off the CUDA cores
// that bound those cases; over 4-bit caches the score product has the keys as its
// rows (S^T = K Q^T; see Kv4Slice).
//
// Merge. The part of a unit a CTA covers ("segment") ends with a cross-warp merge
// in shared memory. A unit covered by one CTA is written out directly; otherwise
// each segment stores (o, max, sum) in the workspace and a second kernel, launched as
// the decode's programmatic dependent, merges them once the decode grid is done:
//     O = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s,
// the merge the vLLM Dual Chunk Attention pull request applies to its partial
// softmax outputs. No counters, atomics or fences: the grid boundary orders the
// partials before the merge, whose CTAs are already resident and waiting.
#include <type_traits>

#include "duo_device.cuh"

namespace duo {
namespace {

__device__ unsigned int g_decode_err;

constexpr int kTK = kDecodeTK;  // keys per tile
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kKPW = kTK / kWarps;  // keys of a tile per warp
constexpr int kNSW = 3;             // pipeline stages per warp
// query heads per KV head from which bf16 decode runs its slices on the tensor cores
// (4-bit caches always do)
constexpr int kMmaMinG = 4;

constexpr int ilog2(int v) { return v <= 1 ? 0 : 1 + ilog2(v / 2); }

// Kernel variants, compiled separately so that the paged paths leave the register
// allocation of the kernels that do not use them untouched.
constexpr int kModePlain = 0;  // contiguous retrieval caches, ring caches for streaming heads
constexpr int kModePaged = 1;  // retrieval caches in a paged pool (block table), ring caches
constexpr int kModePool = 2;   // both head kinds in the paged pool
constexpr int kModeDca = 3;    // Dual Chunk Attention: the query vector depends on the key's chunk
constexpr int kModeKv4 = 4;    // 4-bit caches: codes + fp16 (scale, zero) per row
constexpr int kModeKv4Paged = 5;  // 4-bit caches, retrieval rows in a paged pool of blocks

// retrieval caches (and maybe streaming ones) in the paged pool
__host__ __device__ constexpr bool is_paged_mode(int mode) { return mode == kModePaged || mode == kModePool; }
// 4-bit caches (contiguous or paged retrieval rows)
__host__ __device__ constexpr bool is_kv4_mode(int mode) { return mode == kModeKv4 || mode == kModeKv4Paged; }

template <int D, int G, bool KV4 = false>
struct Cfg {
  static constexpr int DPL = (G * 16 <= 64) ? 16 : 8;  // dims per lane
  static constexpr int LPK = D / DPL;                  // lanes per key
  static constexpr int LB = ilog2(LPK);                // lane bits within a key group
  static constexpr int GB = ilog2(G);                  // head bits
  static constexpr int KPI = 32 / LPK;                 // keys per warp iteration
  static constexpr int IT = kKPW / KPI;                // iterations per tile
  static constexpr int CH = DPL / 8;                   // 16-byte chunks per lane
  // 4-bit caches: tiles of 256 keys, 32 per warp (two 16-key tensor-core groups per
  // slice, so the per-slice costs -- copies, waits, cursor, softmax bookkeeping -- are
  // paid once per 32 keys); two CTAs share an SM, so each warp keeps 2 stages
  static constexpr int KPW = KV4 ? kDecodeTKKv4 / kWarps : kKPW;  // keys of a tile per warp
  static constexpr int TK = KPW * kWarps;              // keys per tile
  static constexpr int NSW = KV4 ? 2 : kNSW;           // pipeline stages per warp
  static constexpr int ROW = KV4 ? D / 2 : D * 2;      // bytes per key row (codes or bf16)
  static constexpr int SLICE = KPW * ROW;              // one warp's K (or V) rows of a tile
  static constexpr int PSLICE = KV4 ? KPW * 4 : 0;     // their (scale, zero) pairs
  static constexpr int WSTAGE = 2 * SLICE + 2 * PSLICE;  // K, V (then K, V pairs)
  static constexpr int RING = kWarps * NSW * WSTAGE;
  static constexpr int RED = kWarps * G * (D + 2);
  static constexpr int PS = D + 4;  // floats per head of a partial in the workspace (16-byte multiple)
  // after the reduction buffer: NSW mbarriers per warp, the segment barrier
  static constexpr size_t SMEM = (size_t)RING + (size_t)RED * 4 + (KV4 ? kWarps * NSW * 8 + 256 : 512);
  static_assert(IT >= 1 && kKPW % KPI == 0, "tile split");
  static_assert(G <= LPK, "every head needs a lane of each key group");
};

struct Unit {
  int b, kvh;
  int64_t plane;  // retrieval: b * n_ret + ri (its row map in the cache)
  bool streaming;
  int64_t keys;  // keys this unit holds
  int64_t pq;    // position of the query
  int64_t ntiles;
  const uint16_t* kb;
  const uint16_t* vb;
};

// CTA whose share of the retrieval tiles contains tile t (shares are [c W / Cr, (c + 1) W / Cr)).
__device__ __forceinline__ int cta_of(const DecodeParams& p, int64_t t) {
  return (int)(((t + 1) * p.Cr - 1) / p.W);
}

// Tokens held by sequence b: the uniform n, or its entry of the device length
// array clamped to the planned maximum n (so no tile beyond the plan is read).
__device__ __forceinline__ int64_t seq_len(const DecodeParams& p, int b) {
  if (!p.seq_lens) return p.n;
  const int64_t v = __ldg(p.seq_lens + b);
  return v < 0 ? 0 : (v > p.n ? p.n : v);
}

// kModePool: streaming heads live in the pool, rows = positions.
template <int kMode>
__device__ __forceinline__ Unit unit_info(const DecodeParams& p, int u) {
  Unit x;
  const int D = p.sh.D;
  if (u < p.U_r) {
    const int ri = u % p.sh.n_ret;
    x.b = u / p.sh.n_ret;
    x.plane = u;
    x.kvh = p.heads.ret_head[ri];
    x.streaming = false;
    x.pq = seq_len(p, x.b) - 1;
    x.keys = x.pq + 1;
    x.ntiles = p.tiles_r;
    const int64_t off = ((int64_t)x.b * p.sh.n_ret + ri) * p.sh.cap * D;
    x.kb = p.k_full + off;
    x.vb = p.v_full + off;
  } else {
    const int us = u - p.U_r;
    const int si = us % p.sh.n_str;
    x.b = us / p.sh.n_str;
    x.plane = -1;
    x.kvh = p.heads.str_head[si];
    x.streaming = true;
    x.pq = seq_len(p, x.b) - 1;
    x.keys = x.pq + 1 < (int64_t)(p.sh.S + p.sh.R) ? x.pq + 1 : (int64_t)(p.sh.S + p.sh.R);
    if (is_kv4_mode(kMode)) x.plane = us;  // its ring plane in the 4-bit arrays
    if (kMode == kModePool) {  // rows [0, n) of its pool blocks, of which only some tiles are read
      x.plane = us;
      x.keys = x.pq + 1;
    }
    x.ntiles = p.tiles_s;
    const int64_t off = ((int64_t)x.b * p.sh.n_str + si) * (int64_t)(p.sh.S + p.sh.R) * D;
    x.kb = p.k_sr + off;
    x.vb = p.v_sr + off;
  }
  return x;
}

// Rows of local tile `lt` (KPW keys per warp) of a unit with `keys` keys that belong to warp w.
template <int KPW = kKPW>
__device__ __forceinline__ int warp_rows(int64_t keys, int64_t lt, int w) {
  const int64_t r = keys - lt * (KPW * kWarps) - (int64_t)w * KPW;
  return r <= 0 ? 0 : (r >= KPW ? KPW : (int)r);
}

// The work of CTA c, in order: its share [t0, t1) of the retrieval tiles (cut into
// segments at unit boundaries), then streaming units c', c' + C, c' + 2C, ... whole,
// c' = (c - s_first) mod C (short caches deal them to the CTAs after the retrieval ones).
// Dealing the short streaming units round-robin keeps their fixed per-segment
// cost (q load, merges) from piling up on the last CTAs.
struct SegState {
  int64_t rt;  // next retrieval tile
  int k;       // next streaming unit ordinal of this CTA
};

__device__ __forceinline__ bool next_segment(const DecodeParams& p, int c, int64_t t1, bool streaming_too,
                                             SegState& st, int& u, int64_t& lt0, int64_t& lt1) {
  if (st.rt < t1) {
    u = (int)(st.rt / p.tiles_r);  // once per segment
    const int64_t us = (int64_t)u * p.tiles_r;
    const int64_t te = us + p.tiles_r < t1 ? us + p.tiles_r : t1;
    lt0 = st.rt - us;
    lt1 = te - us;
    st.rt = te;
    return true;
  }
  const int64_t sidx = (c >= p.s_first ? c - p.s_first : c + p.C - p.s_first) + (int64_t)st.k * p.C;
  if (streaming_too && sidx < p.U_s) {
    u = p.U_r + (int)sidx;
    lt0 = 0;
    lt1 = p.tiles_s;
    ++st.k;
    return true;
  }
  return false;
}

// Row tile read at local tile lt of a streaming unit kept in the pool: its sink
// tiles, then the window tiles that are not among them.
__device__ __forceinline__ int64_t stream_tile(const DecodeParams& p, int64_t lt) {
  return lt < p.s_sink_tiles ? lt : p.s_win_lo + (lt - p.s_sink_tiles);
}

// The tile this warp refills next, walked forward one tile at a time. With a paged
// pool (kModePaged, kModePool) the cursor also tracks the pool block of its tile: the eight warp
// slices of a tile lie in one block (block sizes are multiples of kTK), so for a
// retrieval unit the block table is read only when the cursor enters a new block, one
// tile before the copy is issued, and a division is needed only where a segment
// starts. The few tiles of a streaming unit in the pool are located one by one.
template <int kMode>
struct Cursor {
  static constexpr bool kPaged = is_paged_mode(kMode);
  SegState st;
  int u;
  int64_t lt, lt1;
  Unit x;
  bool live;
  int tpb;  // paged: tiles per block
  int bi;   // paged: index of the block holding the tile in the unit's table row
  int bt;   // paged: the tile's index within that block
  int blk;  // paged: the block id there (as stored, unchecked)
  // 4-bit retrieval rows in a pool (lane 0 only): the (plane, block index) whose id is in
  // kv4_blk, and the id of the block after it, loaded ahead so that its latency passes
  // while the slices of the current block are consumed
  int kv4_plane = -1, kv4_bi = -1, kv4_blk = 0, kv4_next = 0;
  __device__ __forceinline__ bool in_pool() const { return !x.streaming || kMode == kModePool; }
  // row tile of the current position (= lt except for a streaming unit in the pool)
  __device__ __forceinline__ int64_t row_tile() const { return (int64_t)bi * tpb + bt; }
  __device__ __forceinline__ void fetch_block(const DecodeParams& p) {
    // tiles past the keys are never read (their table entry may not exist)
    if ((kMode == kModePool ? row_tile() : lt) * kTK < x.keys)
      blk = ((kMode == kModePool && x.streaming) ? p.pg.stream_table : p.pg.table)[x.plane * p.pg.max_blocks + bi];
  }
  __device__ __forceinline__ void locate(const DecodeParams& p) {
    if (live && in_pool()) {
      // rows stay below block_size x max_blocks < 2^31 (checked on the host)
      const int64_t k = (kMode == kModePool && x.streaming) ? stream_tile(p, lt) : lt;
      bi = (int)((uint32_t)k / (uint32_t)tpb);
      bt = (int)k - bi * tpb;
      fetch_block(p);
    }
  }
  __device__ __forceinline__ void init(const DecodeParams& p, int c, int64_t t0, int64_t t1, bool streaming_too) {
    st.rt = t0;
    st.k = 0;
    live = next_segment(p, c, t1, streaming_too, st, u, lt, lt1);
    if (live) x = unit_info<kMode>(p, u);
    if (kPaged) {
      tpb = p.pg.block_size / kTK;
      bi = bt = blk = 0;
      locate(p);
    }
  }
  __device__ __forceinline__ void advance(const DecodeParams& p, int c, int64_t t1, bool streaming_too) {
    if (++lt == lt1) {
      live = next_segment(p, c, t1, streaming_too, st, u, lt, lt1);
      if (live) x = unit_info<kMode>(p, u);
      if (kPaged) locate(p);
    } else if (kPaged && !x.streaming) {
      if (++bt == tpb) {
        bt = 0;
        ++bi;
        fetch_block(p);
      }
    } else if (kMode == kModePool) {
      locate(p);
    }
  }
};

// Copies this warp's slice of the cursor's tile into a stage, under the L2 policy pol.
// Returns true when the slice lies in a paged block whose id is out of range: then
// nothing is copied, the error is recorded and the consumer skips the slice's rows.
template <int D, int G, int kMode>
__device__ __forceinline__ bool issue_slice(const DecodeParams& p, Cursor<kMode>& cur, int w,
                                            uint8_t* stage, uint64_t* bar, uint64_t pol) {
  using C = Cfg<D, G, is_kv4_mode(kMode)>;
  if constexpr (is_kv4_mode(kMode)) {
    // the slice's rows rounded up to whole 16-row groups of codes and (scale, zero)
    // pairs: the planes' row pitches are multiples of 16, so the groups stay inside
    // their plane; rows past the keys are copied but never used
    const int rows = warp_rows<C::KPW>(cur.x.keys, cur.lt, w);
    if (rows <= 0) {
      mbar_arrive_expect_tx(bar, 0);
      return false;
    }
    const uint32_t r16 = (uint32_t)(rows + 15) & ~15u;
    int64_t r = cur.x.plane * (cur.x.streaming ? (int64_t)p.sr16 : p.cap16) + cur.lt * C::TK + (int64_t)w * C::KPW;
    if (kMode == kModeKv4Paged && !cur.x.streaming) {
      // the slice's 32 rows lie in one block (block sizes are multiples of 128)
      // rows stay below block_size x max_blocks < 2^31 (checked on the host)
      const int row = (int)(cur.lt * C::TK) + w * C::KPW;
      const int bi = (int)((uint32_t)row / (uint32_t)p.pg.block_size);
      const int plane = (int)cur.x.plane;
      if (plane != cur.kv4_plane || bi != cur.kv4_bi) {
        const int32_t* trow = p.pg.table + (int64_t)plane * p.pg.max_blocks;
        cur.kv4_blk = (plane == cur.kv4_plane && bi == cur.kv4_bi + 1) ? cur.kv4_next : __ldg(trow + bi);
        cur.kv4_plane = plane;
        cur.kv4_bi = bi;
        // the next block's id, if the unit has rows there (else its entry may not exist)
        if ((int64_t)(bi + 1) * p.pg.block_size < cur.x.keys) cur.kv4_next = __ldg(trow + bi + 1);
      }
      const int64_t blk = cur.kv4_blk;
      if (blk < 0 || blk >= p.pg.num_blocks) {
        atomicOr(&g_decode_err, kErrBadBlock);
        mbar_arrive_expect_tx(bar, 0);
        return true;  // nothing copied; the consumer skips the slice's rows
      }
      r = blk * p.pg.block_size + (row - bi * p.pg.block_size);
    }
    const uint8_t* kc = (cur.x.streaming ? p.ks4 : p.k4) + r * (D / 2);
    const uint8_t* vc = (cur.x.streaming ? p.vs4 : p.v4) + r * (D / 2);
    const uint32_t* kz = (cur.x.streaming ? p.kssz : p.ksz) + r;
    const uint32_t* vz = (cur.x.streaming ? p.vssz : p.vsz) + r;
    mbar_arrive_expect_tx(bar, r16 * (2 * C::ROW + 8));
    bulk_g2s_hint(stage, kc, r16 * C::ROW, bar, pol);
    bulk_g2s_hint(stage + C::SLICE, vc, r16 * C::ROW, bar, pol);
    bulk_g2s_hint(stage + 2 * C::SLICE, kz, r16 * 4, bar, pol);
    bulk_g2s_hint(stage + 2 * C::SLICE + C::PSLICE, vz, r16 * 4, bar, pol);
    return false;
  }
  const bool pool = is_paged_mode(kMode) && cur.in_pool();
  int rows = warp_rows(cur.x.keys, kMode == kModePool ? cur.row_tile() : cur.lt, w);
  const uint16_t* kp;
  const uint16_t* vp;
  bool bad = false;
  if (pool) {
    if (rows > 0 && (cur.blk < 0 || cur.blk >= p.pg.num_blocks)) {
      atomicOr(&g_decode_err, kErrBadBlock);
      rows = 0;
      bad = true;
    }
    const int64_t off = ((int64_t)cur.blk * p.pg.block_size + cur.bt * kTK + w * kKPW) * D;
    kp = p.k_full + off;
    vp = p.v_full + off;
  } else {
    const int64_t row0 = cur.lt * kTK + (int64_t)w * kKPW;
    kp = cur.x.kb + row0 * D;
    vp = cur.x.vb + row0 * D;
  }
  const uint32_t bytes = (uint32_t)rows * C::ROW;
  mbar_arrive_expect_tx(bar, 2 * bytes);
  if (rows > 0) {
    bulk_g2s_hint(stage, kp, bytes, bar, pol);
    bulk_g2s_hint(stage + C::SLICE, vp, bytes, bar, pol);
  }
  return bad;
}

__device__ __forceinline__ float2 unpack2(uint32_t w) { return make_float2(bf16lo(w), bf16hi(w)); }

// fp16 (scale, zero) pair of a 4-bit row, widened to fp32
__device__ __forceinline__ float2 scale_zero(uint32_t w) {
  return make_float2(__half2float(__ushort_as_half((unsigned short)(w & 0xFFFFu))),
                     __half2float(__ushort_as_half((unsigned short)(w >> 16))));
}

// ------------------------------------------------------------ warp-MMA consumer
// Warp-level m16n8k16 tensor-core MMA with fp32 accumulation (A row-major, B
// column-major). Fragment layout (lane = 4 gid + tig): a0 (row gid, cols 2 tig, +1),
// a1 (row gid + 8, same cols), a2 (row gid, cols 2 tig + 8, +9), a3 (row gid + 8,
// cols 2 tig + 8, +9); b0 (rows 2 tig, +1, col gid), b1 (rows 2 tig + 8, +9, col
// gid); c0 c1 (row gid, cols 2 tig, +1), c2 c3 (row gid + 8, same cols); the lower
// column (row) index sits in the low 16 bits of a register.
template <bool F16>
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  if constexpr (F16) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// 4-bit codes as fp16 without a conversion instruction: a code c in bits 0-3 of a
// 16-bit half under the exponent of 1024 (0x6400) reads as 1024 + c, a code in bits
// 4-7 under the exponent of 64 (0x5400, unit in the last place 1/16) as 64 + c.
constexpr uint32_t kLoMagic = 0x64006400u, kHiMagic = 0x54005400u;

// (x & mask) | magic in one instruction
__device__ __forceinline__ uint32_t and_or(uint32_t x, uint32_t mask, uint32_t magic) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(x), "r"(mask), "r"(magic));
  return d;
}

// The per-warp consumer of bf16 caches used when the query heads of a KV head are
// many: a warp's 16-key slice is two tensor-core products instead of one packed FMA
// per (element, head pair).
//   S = Q K^T   rows = the g query heads (rows g ... 15 zero), cols = 8 keys per
//               n-tile (keys gid and gid + 8 are the columns lane gid loads), k = dims
//   O^T += V^T P^T   rows = 16 dims per m-tile, cols = the heads, k = the 16 keys
// The dims inside a k-step may be taken in any order as long as Q and K use the same
// one, and the rows of O^T in any order as long as the output is written back with
// it; both orders below are chosen so that each lane reads whole 16-byte pieces of
// shared memory and needs no shuffles to build its fragments:
//   K: k-step 2u + e, k-index 2 tig + i (+ 8) <-> dim 8 (tig + 4u) + 4e + i (+ 2)
//   O^T: m-tile i, row gid (gid + 8) <-> dim (D / 8) gid + 2i (+ 1)
// After S the softmax of the slice runs in the accumulator layout: lane (gid, tig)
// holds head gid's scores of keys 2 tig, 2 tig + 1, 2 tig + 8, 2 tig + 9, which are
// exactly the keys of its P^T fragment.
// One slice as the consumer sees it: its K and V rows (codes) in shared memory, for
// 4-bit caches their (scale, zero) pairs, and the bits of the slice's values (key_of
// of each consumer gives their keys) that hold a visible key (hvalid: the same,
// cleared on the values of heads >= G).
struct SliceIn {
  const uint8_t* k;
  const uint8_t* v;
  const uint8_t* kz;
  const uint8_t* vz;
  uint32_t kvalid, hvalid;
};

struct NoMma {};  // stands in for the warp-MMA consumers in the kernels that do not use them

template <int D, int G>
struct MmaSlice {
  static constexpr int KS = D / 16;   // k-steps of S over the dims
  static constexpr int MT = D / 16;   // 16-dim m-tiles of O^T
  static constexpr int DT = D / 8;    // output dims of a lane: DT gid ... DT gid + DT - 1
  static constexpr int ROW = D * 2;   // bytes per row
  uint32_t qa[KS][2];  // a0, a2 of every k-step (a1 = a3 = 0: rows 8 ... 15)
  float o[MT][4];
  float m_run, l_part, qfac;

  // value k of a slice (0 ... 3): key 2 tig + k % 2 + 8 (k / 2), head gid
  __device__ static __forceinline__ int key_of(int k, int, int tig) { return 2 * tig + (k & 1) + 8 * ((k >> 1) & 1); }
  __device__ static __forceinline__ uint32_t head_mask(uint32_t kvalid, int gid, int) { return gid < G ? kvalid : 0u; }

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int i = 0; i < MT; ++i)
#pragma unroll
      for (int k = 0; k < 4; ++k) o[i][k] = 0.f;
    m_run = -INFINITY;
    l_part = 0.f;
  }

  // q row of head gid (nullptr for the zero rows gid >= G) into A fragments; factor is
  // the softmax scale (times the DCA mscale) applied to the fp32 product
  __device__ __forceinline__ void load_q(const uint16_t* qh, float factor, int tig) {
    qfac = factor;
#pragma unroll
    for (int u = 0; u < D / 32; ++u) {
      const uint4 v = qh ? __ldg(reinterpret_cast<const uint4*>(qh + (tig + 4 * u) * 8)) : make_uint4(0, 0, 0, 0);
      qa[2 * u][0] = v.x;
      qa[2 * u][1] = v.y;
      qa[2 * u + 1][0] = v.z;
      qa[2 * u + 1][1] = v.w;
    }
  }

  // One 16-key slice. kFull: every key of the slice is a stored, visible key (an
  // interior tile of a retrieval unit), so no key needs masking; the rows gid >= G then
  // hold finite values for heads that do not exist, whose columns of O^T are never
  // written out.
  template <bool kFull>
  __device__ __forceinline__ void slice(const SliceIn& in, int gid, int tig) {
    // x[k]: scores of keys 2 tig, 2 tig + 1, 2 tig + 8, 2 tig + 9
    float x[4];
    float sc[2][2][4];  // [n-tile][chain][fragment]: two independent accumulation chains
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int k = 0; k < 4; ++k) sc[j][c][k] = 0.f;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint8_t* row = in.k + (gid + 8 * j) * ROW;
#pragma unroll
      for (int u = 0; u < D / 32; ++u) {
        const uint4 v = *reinterpret_cast<const uint4*>(row + (tig + 4 * u) * 16);
        mma16816<false>(sc[j][u & 1], qa[2 * u][0], 0u, qa[2 * u][1], 0u, v.x, v.y);
        mma16816<false>(sc[j][u & 1], qa[2 * u + 1][0], 0u, qa[2 * u + 1][1], 0u, v.z, v.w);
      }
    }
    x[0] = sc[0][0][0] + sc[0][1][0];
    x[1] = sc[0][0][1] + sc[0][1][1];
    x[2] = sc[1][0][0] + sc[1][1][0];
    x[3] = sc[1][0][1] + sc[1][1][1];
    float mx = -INFINITY;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      x[k] = (kFull || ((in.hvalid >> k) & 1u)) ? x[k] * qfac : -INFINITY;
      mx = fmaxf(mx, x[k]);
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const bool grow = mx > m_run + 8.f;  // lazy rescale, as in the CUDA-core path
    if (__any_sync(0xffffffffu, grow)) {
      const float f = grow ? ex2_approx(m_run - mx) : 1.f;
      if (grow) {
        m_run = mx;
        l_part *= f;
      }
      const float f0 = __shfl_sync(0xffffffffu, f, 8 * tig);      // head 2 tig
      const float f1 = __shfl_sync(0xffffffffu, f, 8 * tig + 4);  // head 2 tig + 1
#pragma unroll
      for (int i = 0; i < MT; ++i) {
        o[i][0] *= f0;
        o[i][1] *= f1;
        o[i][2] *= f0;
        o[i][3] *= f1;
      }
    }
    float pr[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      pr[k] = (kFull || ((in.hvalid >> k) & 1u)) ? ex2_approx(x[k] - m_run) : 0.f;
      l_part += pr[k];
    }
    const int kr[4] = {2 * tig, 2 * tig + 1, 2 * tig + 8, 2 * tig + 9};
    const uint32_t pb0 = pack_bf16x2(pr[0], pr[1]);
    const uint32_t pb1 = pack_bf16x2(pr[2], pr[3]);
    uint32_t w[4][MT];  // MT words = this lane's DT dims of each key
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const bool ok = kFull || ((in.kvalid >> k) & 1u);  // rows not copied in this stage may hold anything
#pragma unroll
      for (int c = 0; c < MT / 4; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(in.v + kr[k] * ROW + DT * 2 * gid + c * 16);
        w[k][4 * c] = ok ? v.x : 0u;
        w[k][4 * c + 1] = ok ? v.y : 0u;
        w[k][4 * c + 2] = ok ? v.z : 0u;
        w[k][4 * c + 3] = ok ? v.w : 0u;
      }
    }
#pragma unroll
    for (int i = 0; i < MT; ++i)
      mma16816<false>(o[i], __byte_perm(w[0][i], w[1][i], 0x5410), __byte_perm(w[0][i], w[1][i], 0x7632),
                      __byte_perm(w[2][i], w[3][i], 0x5410), __byte_perm(w[2][i], w[3][i], 0x7632), pb0, pb1);
  }

  // The warp's (o, max, sum) per head into the reduction buffer, as the CUDA-core path
  // leaves them: red[(warp G + h) (D + 2) + d], then max and sum at D and D + 1.
  __device__ __forceinline__ void write(float* red, int warp, int gid, int tig) {
    float l = l_part;
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    const int h0 = 2 * tig, h1 = 2 * tig + 1;
#pragma unroll
    for (int i = 0; i < MT; ++i) {
      const int d = DT * gid + 2 * i;
      if (h0 < G) {
        float* r = red + (warp * G + h0) * (D + 2) + d;
        r[0] = o[i][0];
        r[1] = o[i][2];
      }
      if (h1 < G) {
        float* r = red + (warp * G + h1) * (D + 2) + d;
        r[0] = o[i][1];
        r[1] = o[i][3];
      }
    }
    if (tig == 0 && gid < G) {
      float* r = red + (warp * G + gid) * (D + 2);
      r[D] = m_run;
      r[D + 1] = l;
    }
  }
};

// 8x8 transpose of a b16 matrix held in fragment layout (lane 4 gid + tig holds row
// gid, cols 2 tig and 2 tig + 1); afterwards the lane holds row gid of the transpose.
__device__ __forceinline__ uint32_t transpose8x8(uint32_t m) {
  uint32_t d;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(m));
  return d;
}

// The consumer over 4-bit caches: a warp's slice is 32 keys, two 16-key groups, and
// the score product has the keys, not the heads, as its rows:
//   S^T = K Q^T   rows = the 16 keys of a group, cols = the query heads (8 columns, g
//                 of them real), k = dims
//   O^T += V^T P^T   rows = 16 dims per m-tile, cols = the heads, k = the 16 keys
// The K codes form the A fragments: lane (gid, tig) reads code words w = (D / 32) tig
// + u (dims 8w ... 8w + 7) of keys 16 q + gid and 16 q + gid + 8, with k-step 2u + e,
// k-index 2 tig + i (+ 8) <-> dim 8w + 2e + 4i (+ 1); q, rounded to fp16, forms the B
// fragments in the same order. That is sixteen products per 32 keys, none spent on
// zero rows, and no zero registers beside q. The codes become fp16 by bit placement
// (kLoMagic, kHiMagic); their offsets are folded into one constant per head (sum of q
// times the offsets of its dims), removed from each slice's fresh fp32 accumulator, so
// that q.k^ = scale (q.c) + zero sum(q). Lane (gid, tig) then holds the scores of keys
// gid and gid + 8 of each group for heads 2 tig and 2 tig + 1: the running max, sum and
// zero sum of those two heads live in the lane, and the rescale of its O^T columns (the
// same two heads) needs no shuffle. P^T is made from the scores with one 8x8 transpose
// per 8 keys. The V codes enter as fp16 subnormals, masked out of the word with no
// offset (c 2^-24 from bits 0-3, c 2^-20 from bits 4-7; exact), so the long-lived O
// accumulator carries no offset and each output dim comes back with its power of two
// (O^T rows as in MmaSlice); p v^ = (p scale) c + p zero with p scale rounded to fp16
// and the zero part summed per head in fp32. q goes through fp16 on this path, so its
// values must lie within the fp16 range (bf16 values there convert exactly).
template <int D, int G>
struct Kv4Slice {
  static constexpr int KS = D / 16;  // k-steps of S over the dims
  static constexpr int MT = D / 16;  // 16-dim m-tiles of O^T
  static constexpr int DT = D / 8;   // output dims of a lane: DT gid ... DT gid + DT - 1
  static constexpr int ROW = D / 2;  // code bytes per row
  static constexpr int WPT = D / 32;  // code words of a lane per K row
  static constexpr int NGRP = 2;     // 16-key groups per 32-key slice
  // p (at most 2^8 under the lazy rescale) times the row scale enters the V product in
  // fp16 as p scale 2^-6, so that no row within the fp16 range can overflow it; the V
  // codes enter as subnormals, c 2^-24 (even dims) and c 2^-20 (odd dims)
  static constexpr float kOScale = 64.f, kVLo = 16777216.f, kVHi = 1048576.f;
  uint32_t qb[KS][2];  // b0, b1 of every k-step: head gid's q at k-indices 2 tig (+1), 2 tig + 8 (+9)
  float o[MT][4];
  float m_run[2], l_part[2], z_part[2];  // heads 2 tig, 2 tig + 1
  float off[2], qsum[2];                 // their folded offsets and sums of q
  float qfac;

  // value k of a slice (0 ... 7): key 16 (k / 4) + gid + 8 ((k / 2) % 2), head 2 tig + k % 2
  __device__ static __forceinline__ int key_of(int k, int gid, int) { return 16 * (k >> 2) + gid + 8 * ((k >> 1) & 1); }
  __device__ static __forceinline__ uint32_t head_mask(uint32_t kvalid, int, int tig) {
    return kvalid & ((2 * tig < G ? 0x55u : 0u) | (2 * tig + 1 < G ? 0xAAu : 0u));
  }

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int i = 0; i < MT; ++i)
#pragma unroll
      for (int k = 0; k < 4; ++k) o[i][k] = 0.f;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      m_run[e] = -INFINITY;
      l_part[e] = 0.f;
      z_part[e] = 0.f;
    }
  }

  // q row of head gid (nullptr for the heads gid >= G) into B fragments, rounded to fp16
  __device__ __forceinline__ void load_q(const uint16_t* qh, float factor, int tig) {
    qfac = factor;
    float so = 0.f, ss = 0.f;
#pragma unroll
    for (int u = 0; u < WPT; ++u) {
      const int w = WPT * tig + u;
      const uint4 v = qh ? __ldg(reinterpret_cast<const uint4*>(qh + w * 8)) : make_uint4(0, 0, 0, 0);
      const uint32_t b[4] = {v.x, v.y, v.z, v.w};
      float h[8];  // dims 8w ... 8w + 7 rounded to fp16 (exact for bf16 values in its range)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        h[2 * k] = __half2float(__float2half_rn(bf16lo(b[k])));
        h[2 * k + 1] = __half2float(__float2half_rn(bf16hi(b[k])));
      }
      qb[2 * u][0] = pack_half2(h[0], h[4]);
      qb[2 * u][1] = pack_half2(h[1], h[5]);
      qb[2 * u + 1][0] = pack_half2(h[2], h[6]);
      qb[2 * u + 1][1] = pack_half2(h[3], h[7]);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        ss += h[k];
        so = fmaf(h[k], (k & 1) ? 64.f : 1024.f, so);
      }
    }
#pragma unroll
    for (int m = 1; m <= 2; m <<= 1) {
      ss += __shfl_xor_sync(0xffffffffu, ss, m);
      so += __shfl_xor_sync(0xffffffffu, so, m);
    }
    // lanes 4 h hold head h's sums; this lane wants heads 2 tig and 2 tig + 1
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      off[e] = __shfl_sync(0xffffffffu, so, 4 * (2 * tig + e));
      qsum[e] = __shfl_sync(0xffffffffu, ss, 4 * (2 * tig + e));
    }
  }

  // One 32-key slice (two 16-key groups). kFull: every key is a stored, visible key of
  // an interior tile; the columns of heads >= G then hold finite values never written out.
  template <bool kFull>
  __device__ __forceinline__ void slice(const SliceIn& in, int gid, int tig) {
    // x[4 q + k]: (key a, head 2 tig), (a, 2 tig + 1), (key b, 2 tig), (b, 2 tig + 1)
    // with a = 16 q + gid, b = a + 8
    float x[4 * NGRP];
#pragma unroll
    for (int q = 0; q < NGRP; ++q) {
      float sc[2][4];  // even and odd k-steps: two independent accumulation chains
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int k = 0; k < 4; ++k) sc[c][k] = 0.f;
      uint32_t wa[WPT], wb[WPT];  // lane tig: words WPT tig ... of rows a and b
      const uint8_t* ra = in.k + (16 * q + gid) * ROW;
      const uint8_t* rb = ra + 8 * ROW;
      if constexpr (WPT == 4) {
        const uint4 va = *reinterpret_cast<const uint4*>(ra + tig * 16);
        const uint4 vb = *reinterpret_cast<const uint4*>(rb + tig * 16);
        wa[0] = va.x, wa[1] = va.y, wa[2] = va.z, wa[3] = va.w;
        wb[0] = vb.x, wb[1] = vb.y, wb[2] = vb.z, wb[3] = vb.w;
      } else {
        const uint2 va = *reinterpret_cast<const uint2*>(ra + tig * 8);
        const uint2 vb = *reinterpret_cast<const uint2*>(rb + tig * 8);
        wa[0] = va.x, wa[1] = va.y;
        wb[0] = vb.x, wb[1] = vb.y;
      }
#pragma unroll
      for (int u = 0; u < WPT; ++u) {
        const uint32_t xa = wa[u], xb = wb[u], xa8 = xa >> 8, xb8 = xb >> 8;
        mma16816<true>(sc[0], and_or(xa, 0x000F000Fu, kLoMagic), and_or(xb, 0x000F000Fu, kLoMagic),
                       and_or(xa, 0x00F000F0u, kHiMagic), and_or(xb, 0x00F000F0u, kHiMagic), qb[2 * u][0],
                       qb[2 * u][1]);
        mma16816<true>(sc[1], and_or(xa8, 0x000F000Fu, kLoMagic), and_or(xb8, 0x000F000Fu, kLoMagic),
                       and_or(xa8, 0x00F000F0u, kHiMagic), and_or(xb8, 0x00F000F0u, kHiMagic), qb[2 * u + 1][0],
                       qb[2 * u + 1][1]);
      }
      const float2 sa = scale_zero(*reinterpret_cast<const uint32_t*>(in.kz + 4 * (16 * q + gid)));
      const float2 sb = scale_zero(*reinterpret_cast<const uint32_t*>(in.kz + 4 * (16 * q + 8 + gid)));
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 sz = (k & 2) ? sb : sa;
        const int e = k & 1;
        x[4 * q + k] = fmaf(sz.x, (sc[0][k] + sc[1][k]) - off[e], sz.y * qsum[e]);
      }
    }
    // per head: max over the lane's keys, then over the eight row groups
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int k = 0; k < 4 * NGRP; ++k) {
      x[k] = (kFull || ((in.hvalid >> k) & 1u)) ? x[k] * qfac : -INFINITY;
      mx[k & 1] = fmaxf(mx[k & 1], x[k]);
    }
#pragma unroll
    for (int s = 4; s < 32; s <<= 1)
#pragma unroll
      for (int e = 0; e < 2; ++e) mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], s));
    const bool g0 = mx[0] > m_run[0] + 8.f, g1 = mx[1] > m_run[1] + 8.f;  // lazy rescale
    if (__any_sync(0xffffffffu, g0 || g1)) {
      const float f0 = g0 ? ex2_approx(m_run[0] - mx[0]) : 1.f;
      const float f1 = g1 ? ex2_approx(m_run[1] - mx[1]) : 1.f;
      if (g0) {
        m_run[0] = mx[0];
        l_part[0] *= f0;
        z_part[0] *= f0;
      }
      if (g1) {
        m_run[1] = mx[1];
        l_part[1] *= f1;
        z_part[1] *= f1;
      }
#pragma unroll
      for (int i = 0; i < MT; ++i) {
        o[i][0] *= f0;
        o[i][1] *= f1;
        o[i][2] *= f0;
        o[i][3] *= f1;
      }
    }
#pragma unroll
    for (int q = 0; q < NGRP; ++q) {
      const float2 va = scale_zero(*reinterpret_cast<const uint32_t*>(in.vz + 4 * (16 * q + gid)));
      const float2 vb = scale_zero(*reinterpret_cast<const uint32_t*>(in.vz + 4 * (16 * q + 8 + gid)));
      float b[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 sz = (k & 2) ? vb : va;
        const int e = k & 1;
        const bool ok = kFull || ((in.hvalid >> (4 * q + k)) & 1u);  // an unused row's pair may be anything
        const float pk = ok ? ex2_approx(x[4 * q + k] - m_run[e]) : 0.f;
        l_part[e] += pk;
        b[k] = ok ? pk * (sz.x * (1.f / kOScale)) : 0.f;
        z_part[e] += ok ? pk * sz.y : 0.f;
      }
      // [key][head] rows a and b, transposed to P^T's fragments: keys 2 tig (+1), 2 tig + 8 (+9) of head gid
      const uint32_t pb0 = transpose8x8(pack_half2(b[0], b[1]));
      const uint32_t pb1 = transpose8x8(pack_half2(b[2], b[3]));
      // V codes in fragment order (see the 4-bit append): in group q, the lane's word i
      // holds, for its dims of m-tile i, the codes of keys 2 tig, 2 tig + 8, 2 tig + 1,
      // 2 tig + 9
      uint32_t w[MT];
#pragma unroll
      for (int c = 0; c < MT / 4; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(in.v + 16 * ROW * q + (4 * gid + tig) * MT * 4 + 16 * c);
        w[4 * c] = v.x;
        w[4 * c + 1] = v.y;
        w[4 * c + 2] = v.z;
        w[4 * c + 3] = v.w;
      }
#pragma unroll
      for (int i = 0; i < MT; ++i) {
        const uint32_t x8 = w[i] >> 8;
        // the codes as fp16 subnormals: c 2^-24 (bits 0-3) and c 2^-20 (bits 4-7)
        mma16816<true>(o[i], w[i] & 0x000F000Fu, w[i] & 0x00F000F0u, x8 & 0x000F000Fu, x8 & 0x00F000F0u, pb0,
                       pb1);
      }
    }
  }

  // The warp's (o, max, sum) per head into the reduction buffer: red[(warp G + h) (D + 2)
  // + d], then max and sum at D and D + 1.
  __device__ __forceinline__ void write(float* red, int warp, int gid, int tig) {
    float l[2], z[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      l[e] = l_part[e];
      z[e] = z_part[e];
#pragma unroll
      for (int s = 4; s < 32; s <<= 1) {
        l[e] += __shfl_xor_sync(0xffffffffu, l[e], s);
        z[e] += __shfl_xor_sync(0xffffffffu, z[e], s);
      }
    }
    const int h0 = 2 * tig, h1 = 2 * tig + 1;
#pragma unroll
    for (int i = 0; i < MT; ++i) {
      const int d = DT * gid + 2 * i;
      if (h0 < G) {
        float* r = red + (warp * G + h0) * (D + 2) + d;
        r[0] = fmaf(o[i][0], kOScale * kVLo, z[0]);
        r[1] = fmaf(o[i][2], kOScale * kVHi, z[0]);
      }
      if (h1 < G) {
        float* r = red + (warp * G + h1) * (D + 2) + d;
        r[0] = fmaf(o[i][1], kOScale * kVLo, z[1]);
        r[1] = fmaf(o[i][3], kOScale * kVHi, z[1]);
      }
    }
    if (gid == 0) {
#pragma unroll
      for (int e = 0; e < 2; ++e)
        if (2 * tig + e < G) {
          float* r = red + (warp * G + 2 * tig + e) * (D + 2);
          r[D] = m_run[e];
          r[D + 1] = l[e];
        }
    }
  }
};

// Synchronisation of the eight warps through an mbarrier (bounded wait).
struct WarpSync {
  uint64_t* bar;
  uint32_t phase;
  __device__ __forceinline__ bool sync(DevError err) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
    const bool ok = mbar_wait(bar, phase, err, kErrDecodeConsumer);
    phase ^= 1u;
    __syncwarp();
    return ok;
  }
};

template <int D, int G, int kMode>
__global__ void __launch_bounds__(kThreads, is_kv4_mode(kMode) ? kDecodeCtasPerSmKv4 : 1)
    decode_kernel(const DecodeParams p) {
  using C = Cfg<D, G, is_kv4_mode(kMode)>;
  extern __shared__ __align__(1024) uint8_t smem[];
  float* red = reinterpret_cast<float*>(smem + C::RING);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::RING + (size_t)C::RED * 4);  // [kWarps][C::NSW]
  uint64_t* segbar = full + kWarps * C::NSW;

  const DevError err{&g_decode_err};
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  const int64_t t0 = c < p.Cr ? (int64_t)c * p.W / p.Cr : p.W;
  // After any CTA of this kernel gave up a wait, later CTAs do no work.
  const bool live = *(volatile unsigned int*)err.word == 0u;
  const int64_t t1 = live && c < p.Cr ? (int64_t)(c + 1) * p.W / p.Cr : t0;
  uint8_t* ring = smem + (size_t)warp * C::NSW * C::WSTAGE;
  uint64_t* wfull = full + warp * C::NSW;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kWarps * C::NSW; ++s) mbar_init(&full[s], 1);
    mbar_init(segbar, kWarps);
    fence_mbarrier_init();
  }
  __syncthreads();
  // Launched as a programmatic dependent (of the append before it, say): nothing the
  // previous grid writes (cache rows, ring slots, positions, lengths) is read before it ends.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // The cache rows are read once: L2 lets them go first, keeping q and the partials the
  // merge reads. The merge kernel launched after this one may be scheduled now.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const uint64_t pol = l2_policy_evict_first();
  // refill cursor (warp-uniform); the prologue issues the first C::NSW - 1 slices
  constexpr bool kPaged = is_paged_mode(kMode);
  constexpr bool kBadBlocks = kPaged || kMode == kModeKv4Paged;  // a slice may come from a bad block id
  Cursor<kMode> cur;
  cur.init(p, c, t0, t1, live);
  uint32_t issued = 0;  // slices issued (fewer than 2^32 per CTA)
  uint32_t badmask = 0;  // lane 0: bit s set when stage s holds a skipped (bad-block) slice
  for (int s = 0; s < C::NSW - 1 && cur.live; ++s) {
    if (lane == 0) {
      const bool bad = issue_slice<D, G, kMode>(p, cur, warp, ring + s * C::WSTAGE, &wfull[s], pol);
      if (kBadBlocks) badmask = bad ? (badmask | (1u << s)) : (badmask & ~(1u << s));
    }
    cur.advance(p, c, t1, live);
    ++issued;
  }

  const int kg = lane / C::LPK;           // key within the warp iteration
  const int cl = lane % C::LPK;           // dims slot of this lane within its key group
  const int hme = cl >> (C::LB - C::GB);  // the head this lane ends up owning
  constexpr bool kMma = is_kv4_mode(kMode) || G >= kMmaMinG;
  const int gid = lane >> 2, tig = lane & 3;  // tensor-core slices: fragment row group, thread in group
  using Mma = std::conditional_t<is_kv4_mode(kMode), Kv4Slice<D, G>, MmaSlice<D, G>>;
  std::conditional_t<kMma, Mma, NoMma> mm;
  const int SR = p.sh.S + p.sh.R;
  WarpSync ws{segbar, 0};
  uint32_t j = 0;  // tiles consumed
  bool ok = true;
  SegState seg{t0, 0};
  int u;
  int64_t lt_begin, lt_end;
  while (ok && next_segment(p, c, t1, live, seg, u, lt_begin, lt_end)) {
    const Unit x = unit_info<kMode>(p, u);

    // q of head (hme ^ l) in slot l, this lane's dims, pre-scaled, as fp32 pairs
    float2 q2[G][C::DPL / 2];
    auto load_q = [&](const uint16_t* qsrc, float factor) {
#pragma unroll
      for (int l = 0; l < G; ++l) {
        const uint16_t* qh = qsrc + ((int64_t)x.b * p.sh.Hq + (int64_t)x.kvh * G + (hme ^ l)) * D;
#pragma unroll
        for (int ch = 0; ch < C::CH; ++ch) {
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(qh + (cl + ch * C::LPK) * 8));
          const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = unpack2(w4[e]);
            q2[l][ch * 4 + e] = make_float2(f.x * factor, f.y * factor);
          }
        }
      }
    };
    // DCA: which query vectors the keys of tile lt take (0 query, 1 query_succ for the
    // chunk before the query's, 2 query_inter further back; chunk_len is a multiple of
    // the tile), and the factor: softmax scale times the sequence's fp32 mscale, on fp32 q
    float qfactor = p.scale_log2;
    int qv = 0;
    int64_t t_intra = 0, t_succ = 0;  // first tile of the query's chunk and of the one before
    if (kMode == kModeDca) {
      const int64_t tpc = p.chunk_len / kTK;
      t_intra = (x.pq / p.chunk_len) * tpc;
      t_succ = t_intra - tpc;
    }
    auto dca_var = [&](int64_t lt) { return lt >= t_intra ? 0 : (lt >= t_succ ? 1 : 2); };
    auto dca_q = [&](int v) { return v == 0 ? p.q : (v == 1 ? p.q_succ : p.q_inter); };
    // tensor-core slices: lane (gid, tig) holds head gid's row of the A fragments
    auto set_q = [&](const uint16_t* qsrc) {
      if constexpr (kMma)
        mm.load_q(gid < G ? qsrc + ((int64_t)x.b * p.sh.Hq + (int64_t)x.kvh * G + gid) * D : nullptr, qfactor, tig);
      else
        load_q(qsrc, qfactor);
    };
    if constexpr (kMma) mm.reset();
    if (kMode == kModeDca) {
      if (p.mscale) qfactor *= __ldg(p.mscale + x.b);
      qv = dca_var(lt_begin);
      set_q(dca_q(qv));
    } else {
      set_q(p.q);
    }
    float2 o2[G][C::DPL / 2];
#pragma unroll
    for (int l = 0; l < G; ++l)
#pragma unroll
      for (int e = 0; e < C::DPL / 2; ++e) o2[l][e] = make_float2(0.f, 0.f);
    float l_run = 0.f, m_run = -INFINITY;  // of head hme

    for (int64_t lt = lt_begin; lt < lt_end; ++lt, ++j) {
      const int s = (int)(j % C::NSW);
      if (kMode == kModeDca) {
        const int v = dca_var(lt);
        if (v != qv) {  // at most twice per unit
          qv = v;
          set_q(dca_q(v));
        }
      }
      // refill: the stage used by tile j - 1 is free now (this warp finished it)
      if (cur.live) {
        const int sn = (int)((j + C::NSW - 1) % C::NSW);
        if (lane == 0) {
          const bool bad = issue_slice<D, G, kMode>(p, cur, warp, ring + sn * C::WSTAGE, &wfull[sn], pol);
          if (kBadBlocks) badmask = bad ? (badmask | (1u << sn)) : (badmask & ~(1u << sn));
        }
        cur.advance(p, c, t1, live);
        ++issued;
      }
      if (!mbar_wait(&wfull[s], (uint32_t)((j / C::NSW) & 1), err, kErrDecodeConsumer)) {
        ok = false;
        break;
      }
      // streaming unit in the pool: keys are rows (= positions) of row tile kt
      const bool str_pool = kMode == kModePool && x.streaming;
      const int64_t kt = str_pool ? stream_tile(p, lt) : lt;
      int rows = warp_rows<C::KPW>(x.keys, kt, warp);
      if (kBadBlocks && ((__shfl_sync(0xffffffffu, badmask, 0) >> s) & 1u)) rows = 0;
      const uint8_t* sk = ring + s * C::WSTAGE;
      const uint8_t* sv = sk + C::SLICE;
      const bool full_tile = rows == C::KPW && !x.streaming;

      if constexpr (kMma) {
        // keys 16 q + 2 tig, + 1, + 8, + 9 of the slice's 16-key groups q
        constexpr int NK = 4 * (C::KPW / 16);
        uint32_t kvalid = (1u << NK) - 1u;
        if (!full_tile) {
          kvalid = 0u;
#pragma unroll
          for (int k = 0; k < NK; ++k) {
            const int key = Mma::key_of(k, gid, tig);
            bool valid = key < rows;
            if (x.streaming && valid) {
              const int64_t slot = kt * C::TK + (int64_t)warp * C::KPW + key;
              const int jp = str_pool ? (int)slot : __ldg(p.pos + (int64_t)x.b * SR + slot);
              valid = jp >= 0 && jp <= x.pq && (jp < p.sh.S || x.pq - jp < p.sh.R);
            }
            kvalid |= (uint32_t)valid << k;
          }
        }
        const SliceIn in{sk, sv, sk + 2 * C::SLICE, sk + 2 * C::SLICE + C::PSLICE, kvalid, Mma::head_mask(kvalid, gid, tig)};
        if (full_tile)
          mm.template slice<true>(in, gid, tig);
        else
          mm.template slice<false>(in, gid, tig);
      } else {
        float sc[C::IT];
        bool vis[C::IT];
#pragma unroll
        for (int it = 0; it < C::IT; ++it) {
          const int key = it * C::KPI + kg;  // row within this warp's slice
          bool valid = true;
          if (!full_tile) {
            valid = key < rows;
            if (x.streaming && valid) {
              const int64_t slot = kt * C::TK + (int64_t)warp * C::KPW + key;
              const int jp = str_pool ? (int)slot : __ldg(p.pos + (int64_t)x.b * SR + slot);
              valid = jp >= 0 && jp <= x.pq && (jp < p.sh.S || x.pq - jp < p.sh.R);
            }
          }
          vis[it] = valid;
          float2 acc[G];
#pragma unroll
          for (int l = 0; l < G; ++l) acc[l] = make_float2(0.f, 0.f);
#pragma unroll
          for (int ch = 0; ch < C::CH; ++ch) {
            const uint4 kv = *reinterpret_cast<const uint4*>(sk + key * C::ROW + (cl + ch * C::LPK) * 16);
            const uint32_t w4[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 k2 = unpack2(w4[e]);
#pragma unroll
              for (int l = 0; l < G; ++l) acc[l] = __ffma2_rn(q2[l][ch * 4 + e], k2, acc[l]);
            }
          }
          float dot[G];
#pragma unroll
          for (int l = 0; l < G; ++l) dot[l] = acc[l].x + acc[l].y;
          // reduce-scatter over the high lane bits: keep the low half of the slots
#pragma unroll
          for (int k = 1; k <= C::GB; ++k) {
            const int half = G >> k;
            const int bit = 1 << (C::LB - k);
#pragma unroll
            for (int l = 0; l < half; ++l) dot[l] += __shfl_xor_sync(0xffffffffu, dot[l + half], bit);
          }
          // butterfly over the remaining lane bits
#pragma unroll
          for (int b = C::LB - C::GB - 1; b >= 0; --b) dot[0] += __shfl_xor_sync(0xffffffffu, dot[0], 1 << b);
          sc[it] = valid ? dot[0] : -INFINITY;
        }

        // tile max of this lane's head over the warp, lazy rescale
        float mx = sc[0];
#pragma unroll
        for (int it = 1; it < C::IT; ++it) mx = fmaxf(mx, sc[it]);
#pragma unroll
        for (int off = C::LPK; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const bool grow = mx > m_run + 8.f;
        if (__any_sync(0xffffffffu, grow)) {
          const float f = grow ? ex2_approx(m_run - mx) : 1.f;  // 0 when m was -inf
          if (grow) {
            l_run *= f;
            m_run = mx;
          }
#pragma unroll
          for (int l = 0; l < G; ++l) {
            const float fl = __shfl_xor_sync(0xffffffffu, f, l << (C::LB - C::GB));
            const float2 f2 = make_float2(fl, fl);
#pragma unroll
            for (int e = 0; e < C::DPL / 2; ++e) o2[l][e] = __fmul2_rn(o2[l][e], f2);
          }
        }
#pragma unroll
        for (int it = 0; it < C::IT; ++it) {
          const float pv = vis[it] ? ex2_approx(sc[it] - m_run) : 0.f;
          sc[it] = pv;
          l_run += pv;
        }
#pragma unroll
        for (int it = 0; it < C::IT; ++it) {
          float pl[G];
          pl[0] = sc[it];
#pragma unroll
          for (int l = 1; l < G; ++l) pl[l] = __shfl_xor_sync(0xffffffffu, sc[it], l << (C::LB - C::GB));
          if (full_tile || vis[it]) {
            const int key = it * C::KPI + kg;
#pragma unroll
            for (int ch = 0; ch < C::CH; ++ch) {
              const uint4 vv = *reinterpret_cast<const uint4*>(sv + key * C::ROW + (cl + ch * C::LPK) * 16);
              const uint32_t w4[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 v2 = unpack2(w4[e]);
#pragma unroll
                for (int l = 0; l < G; ++l)
                  o2[l][ch * 4 + e] = __ffma2_rn(make_float2(pl[l], pl[l]), v2, o2[l][ch * 4 + e]);
              }
            }
          }
        }
      }
      __syncwarp();
    }
    if (!ok) break;

    // ---------------------------------------------------- segment merge
    if constexpr (kMma) mm.write(red, warp, gid, tig);
    // sum over the key groups of the warp (each holds other keys)
#pragma unroll
    for (int off = C::LPK; off < 32 && !kMma; off <<= 1) {
      l_run += __shfl_xor_sync(0xffffffffu, l_run, off);
#pragma unroll
      for (int l = 0; l < G; ++l)
#pragma unroll
        for (int e = 0; e < C::DPL / 2; ++e) {
          const float2 o = make_float2(__shfl_xor_sync(0xffffffffu, o2[l][e].x, off),
                                       __shfl_xor_sync(0xffffffffu, o2[l][e].y, off));
          o2[l][e] = __fadd2_rn(o2[l][e], o);
        }
    }
    if (kg == 0 && !kMma) {
#pragma unroll
      for (int l = 0; l < G; ++l) {
        float* r = red + (warp * G + (hme ^ l)) * (D + 2);
#pragma unroll
        for (int ch = 0; ch < C::CH; ++ch)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            r[(cl + ch * C::LPK) * 8 + 2 * e] = o2[l][ch * 4 + e].x;
            r[(cl + ch * C::LPK) * 8 + 2 * e + 1] = o2[l][ch * 4 + e].y;
          }
      }
      if ((cl & ((1 << (C::LB - C::GB)) - 1)) == 0) {  // one lane per head
        float* r = red + (warp * G + hme) * (D + 2);
        r[D] = m_run;
        r[D + 1] = l_run;
      }
    }
    if (!ws.sync(err)) {
      ok = false;
      break;
    }
    const int tid = threadIdx.x;
    // streaming units are whole in one CTA; a retrieval unit spans CTAs c_first ...
    const int64_t us = (int64_t)u * p.tiles_r;
    const int c_first = x.streaming ? c : cta_of(p, us);
    const int n_parts = x.streaming ? 1 : cta_of(p, us + p.tiles_r - 1) - c_first + 1;
    float* part = p.partials + (int64_t)(c + u) * G * C::PS;
    for (int e = tid; e < G * D; e += kThreads) {
      const int h = e / D;
      const int d = e % D;
      float M = -INFINITY;
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red[(w * G + h) * (D + 2) + D]);
      float num = 0.f, den = 0.f;
      for (int w = 0; w < kWarps; ++w) {
        const float* r = red + (w * G + h) * (D + 2);
        const float f = r[D] == -INFINITY ? 0.f : ex2_approx(r[D] - M);
        num = fmaf(f, r[d], num);
        den = fmaf(f, r[D + 1], den);
      }
      if (n_parts == 1) {
        p.o[((int64_t)x.b * p.sh.Hq + (int64_t)x.kvh * G + h) * D + d] =
            __bfloat16_as_ushort(__float2bfloat16_rn(den > 0.f ? num / den : 0.f));
      } else {
        part[h * C::PS + d] = num;
        if (d == 0) {
          part[h * C::PS + D] = M;
          part[h * C::PS + D + 1] = den;
        }
      }
    }
    // the reduction buffer is reused by the next segment
    if (!ws.sync(err)) {
      ok = false;
      break;
    }
  }
  // Copies still in flight (only after an early exit) land before the CTA ends.
  if (lane == 0) {
    for (uint32_t jj = j; jj < issued; ++jj)
      mbar_wait(&wfull[jj % C::NSW], (uint32_t)((jj / C::NSW) & 1), err, kErrDecodeConsumer);
  }
  __syncthreads();
}

// Merge of the retrieval units split over several CTAs, launched right after the decode
// kernel as its programmatic dependent: its CTAs are scheduled while the decode runs
// (the decode signals griddepcontrol.launch_dependents as it starts) and wait in
// griddepcontrol.wait until the decode grid has finished and its partials are visible.
// One CTA per (retrieval unit, head, 32 output dims): lane = output dim, warp w takes
// partials w, w + 8, ..., up to kMergeNB of them per round with all their loads in
// flight, so a unit split over 152 CTAs is merged in one round of loads; the eight
// warps' (max, sum, outputs) are combined through shared memory:
//     O = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s.
constexpr int kMergeWarps = 8;
constexpr int kMergeNB = 20;  // partials in flight per warp

template <int D, int G>
__global__ void __launch_bounds__(kMergeWarps * 32) decode_merge_kernel(const DecodeParams p) {
  constexpr int PS = D + 4;  // floats per head of a partial (Cfg::PS)
  constexpr int DC = D / 32;
  const int dc = blockIdx.x % DC;
  const int h = (blockIdx.x / DC) % G;
  const int u = blockIdx.x / (DC * G);  // retrieval unit
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t us = (int64_t)u * p.tiles_r;
  const int c_first = cta_of(p, us);
  const int n_parts = cta_of(p, us + p.tiles_r - 1) - c_first + 1;
  if (n_parts <= 1) return;  // the decode kernel wrote this unit's output
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int d = dc * 32 + lane;
  float acc = 0.f, den = 0.f, mrun = -INFINITY;
  for (int i0 = warp; i0 < n_parts; i0 += kMergeWarps * kMergeNB) {
    float mb[kMergeNB], lb[kMergeNB], ob[kMergeNB];
#pragma unroll
    for (int i = 0; i < kMergeNB; ++i) {
      const int ii = i0 + i * kMergeWarps;
      if (ii < n_parts) {
        const float* r = p.partials + ((int64_t)(c_first + ii + u) * G + h) * PS;
        mb[i] = __ldcg(r + D);
        lb[i] = __ldcg(r + D + 1);
        ob[i] = __ldcg(r + d);
      } else {
        mb[i] = -INFINITY;
        lb[i] = 0.f;
        ob[i] = 0.f;
      }
    }
    float mnew = mrun;
#pragma unroll
    for (int i = 0; i < kMergeNB; ++i) mnew = fmaxf(mnew, mb[i]);
    if (mnew == -INFINITY) continue;  // no visible key in any partial so far
    const float fo = mrun == -INFINITY ? 0.f : ex2_approx(mrun - mnew);
    den *= fo;
    acc *= fo;
#pragma unroll
    for (int i = 0; i < kMergeNB; ++i) {
      const float f = mb[i] == -INFINITY ? 0.f : ex2_approx(mb[i] - mnew);
      den = fmaf(f, lb[i], den);
      acc = fmaf(f, ob[i], acc);
    }
    mrun = mnew;
  }
  __shared__ float s_acc[kMergeWarps][32];
  __shared__ float s_m[kMergeWarps], s_l[kMergeWarps];
  s_acc[warp][lane] = acc;
  if (lane == 0) {
    s_m[warp] = mrun;
    s_l[warp] = den;
  }
  __syncthreads();
  if (warp == 0) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kMergeWarps; ++w) M = fmaxf(M, s_m[w]);
    float num = 0.f, dsum = 0.f;
#pragma unroll
    for (int w = 0; w < kMergeWarps; ++w) {
      const float f = s_m[w] == -INFINITY ? 0.f : ex2_approx(s_m[w] - M);
      num = fmaf(f, s_acc[w][lane], num);
      dsum = fmaf(f, s_l[w], dsum);
    }
    const int b = u / p.sh.n_ret;
    const int kvh = p.heads.ret_head[u % p.sh.n_ret];
    p.o[((int64_t)b * p.sh.Hq + (int64_t)kvh * G + h) * D + d] =
        __bfloat16_as_ushort(__float2bfloat16_rn(dsum > 0.f ? num / dsum : 0.f));
  }
}

template <int D, int G, int kMode>
cudaError_t launch_v(const DecodeParams& p, cudaStream_t stream) {
  using C = Cfg<D, G, is_kv4_mode(kMode)>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(decode_kernel<D, G, kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  // Programmatic dependents of what precedes them on the stream: the decode's CTAs may be
  // resident before an append before it ends (the decode waits for it first thing; with
  // lengths on the device, measured slower, so not there), the merge's before the decode ends.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.C);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = p.seq_lens ? 0 : 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, decode_kernel<D, G, kMode>, p);
  if (e != cudaSuccess || p.W == 0 || p.Cr == p.U_r) return e;  // no unit split over CTAs
  cfg.gridDim = dim3((unsigned)(p.U_r * G * (D / 32)));
  cfg.blockDim = dim3(kMergeWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_merge_kernel<D, G>, p);
}

// contiguous and paged retrieval caches are separate kernels, so the paged block
// bookkeeping costs the contiguous kernel nothing
template <int D, int G>
cudaError_t launch_t(const DecodeParams& p, cudaStream_t stream) {
  if (p.kv4) return p.pg.table ? launch_v<D, G, kModeKv4Paged>(p, stream) : launch_v<D, G, kModeKv4>(p, stream);
  if (p.chunk_len > 0) return launch_v<D, G, kModeDca>(p, stream);
  if (p.pg.stream_table) return launch_v<D, G, kModePool>(p, stream);
  return p.pg.table ? launch_v<D, G, kModePaged>(p, stream) : launch_v<D, G, kModePlain>(p, stream);
}

}  // namespace

size_t decode_workspace_bytes(const Shape& sh, int num_ctas) {
  const int64_t U = (int64_t)sh.B * sh.Hkv;
  return (size_t)(num_ctas + U) * sh.g * (sh.D + 4) * 4;  // Cfg::PS floats per head and slot
}

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream) {
  const int D = p.sh.D, G = p.sh.g;
  if (D == 128) {
    if (G == 1) return launch_t<128, 1>(p, stream);
    if (G == 2) return launch_t<128, 2>(p, stream);
    if (G == 4) return launch_t<128, 4>(p, stream);
    if (G == 8) return launch_t<128, 8>(p, stream);
  } else if (D == 64) {
    if (G == 1) return launch_t<64, 1>(p, stream);
    if (G == 2) return launch_t<64, 2>(p, stream);
    if (G == 4) return launch_t<64, 4>(p, stream);
    if (G == 8) return launch_t<64, 8>(p, stream);
  }
  return cudaErrorInvalidValue;
}

cudaError_t decode_read_clear_error(uint32_t* code) {
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_decode_err, sizeof(v));
  if (e != cudaSuccess) return e;
  *code = v;
  if (v) {
    v = 0;
    e = cudaMemcpyToSymbol(g_decode_err, &v, sizeof(v));
  }
  return e;
}

}  // namespace duo
