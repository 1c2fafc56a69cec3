// duo_attn_prefill: causal attention of T new tokens for retrieval and streaming
// heads on the fifth-generation tensor cores.
//
// What it computes (DuoAttention README, Abstract): query position i of a
// retrieval head attends to every key j <= i; of a streaming head only to the
// sinks (j < S) and the recent window (i - j < R). Keys come from the cache as
// it was before these tokens (a retrieval head's rows [0, n), a streaming head's
// sink + ring slots with their positions) and from the new tokens themselves, so
// one-shot prefill (n = 0) and each chunk of a chunked prefill against the
// growing cache are the same kernel.
//
// One CTA computes two 128-row query tiles (256 consecutive query rows) of one
// query head, sharing every K and V tile between them (12 warps; setmaxnreg
// moves registers from the TMA/MMA warpgroup to the two softmax warpgroups):
//   warp 8      TMA producer: both Q tiles once, then K and V tiles (128 keys x D,
//               128-byte swizzle) into a 2-stage ring, completion on mbarriers;
//   warp 9      allocates all 512 TMEM columns (per query tile: S, 128 columns,
//               and O, D columns); one thread issues tcgen05.mma in the order
//               S0(j), S1(j), PV0(j), S0(j+1), PV1(j), S1(j+1), ... so the tensor
//               core always has the other tile's work while one softmax runs;
//               P (bf16) overwrites the first 64 columns of its S buffer and is
//               the TMEM A operand of O += P V (V MN-major in shared memory);
//   warps 0-3   softmax of query tile 0, warps 4-7 softmax of query tile 1:
//               thread r owns query row r (TMEM lane r): its whole S row in one
//               TMEM round trip, row max with three-input max, fp32 running max
//               and sum with exp2 and the
//               scale log2(e)/sqrt(D) applied to the fp32 product, O rescaled in
//               TMEM only when the max grows by more than 2^8, P packed to bf16;
//               at the end O / sum is stored as bf16.
// A commit after S_x(j) also covers PV_x(j-1) issued before it, so when the
// softmax sees S_x(j) it may overwrite P_x(j-1) and rescale O_x without waiting
// for anything else.
// KV tiles that no row of the CTA can see are never visited: a streaming head's
// CTA visits the sink tile(s), the ring tiles that can still be visible and the
// <= 5 window tiles instead of all earlier tiles (the block skipping of the
// block-sparse streaming attention the README uses).
#include "duo_device.cuh"

namespace duo {
namespace {

__device__ unsigned int g_prefill_err;

constexpr int BM = kPrefillBM;  // rows per query tile
constexpr int BN = kPrefillBN;  // keys per KV tile
constexpr int kQT = 2;          // query tiles per CTA
constexpr int kRows = BM * kQT;
constexpr int kNS = 2;  // K/V pipeline stages
constexpr int kWarpTma = 8;
constexpr int kWarpMma = 9;
// Threads and register split of an instance. Warpgroups: softmax 0, softmax 1, (TMA, MMA,
// 2 idle) -- the 4-bit instance uses the two idle warps and a fourth warpgroup to
// dequantize its cache tiles (6 warps). The block is launched with kLaunchRegs per
// thread; the warpgroups after the softmax ones drop to kRegsCtl, the softmax
// warpgroups rise to kRegsSoftmax: 2 x 128 x 200 + 128 x 104 = 384 x 168 = 64512, and for
// the 4-bit instance 2 x 128 x 184 + 2 x 128 x 72 = 512 x 128 = 65536, exactly the launch
// totals. The host refuses to launch unless the compiled kernel uses kLaunchRegs.
template <int kMode>
struct Roles;
constexpr uint32_t kTmemCols = 512;
// Kernel variants, compiled separately so that the paged paths leave the register
// allocation of the kernels that do not use them untouched.
constexpr int kModePlain = 0;  // contiguous retrieval caches, ring caches for streaming heads
constexpr int kModePaged = 1;  // retrieval caches in a paged pool (block table), ring caches
constexpr int kModePool = 2;   // both head kinds in the paged pool
constexpr int kModeDca = 3;    // Dual Chunk Attention: one of three query vectors per key tile
constexpr int kModeKv4 = 4;    // 4-bit caches: cache tiles dequantized into shared memory by warps 10, 11
constexpr int kWarpDeq = 10;   // first of the dequantizing warps (4-bit caches): 10 ... 15
template <int kMode>
struct Roles {
  static constexpr bool kKv4 = kMode == kModeKv4;
  static constexpr int kThreads = kKv4 ? 512 : 384;
  static constexpr int kLaunchRegs = kKv4 ? 128 : 168;
  static constexpr int kRegsSoftmax = kKv4 ? 184 : 200;
  static constexpr int kRegsCtl = kKv4 ? 72 : 104;
  static constexpr int kDeqThreads = kThreads - kWarpDeq * 32;  // 4-bit instance: 192
  static_assert(2 * 128 * kRegsSoftmax + (kThreads - 256) * kRegsCtl <= kThreads * kLaunchRegs, "register split");
};
constexpr int kBox = 128 * 128;  // bytes of a 128-row x 64-column bf16 box

__host__ __device__ constexpr uint32_t col_s(int x) { return (uint32_t)x * 256u; }
__host__ __device__ constexpr uint32_t col_o(int x) { return (uint32_t)x * 256u + 128u; }

template <int D>
struct PCfg {
  static constexpr int NBOX = D / 64;
  static constexpr int Q_BYTES = BM * D * 2;  // one query tile
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + kQT * Q_BYTES;
  static constexpr int OFF_V = OFF_K + kNS * KV_BYTES;
  static constexpr int OFF_BAR = OFF_V + kNS * KV_BYTES;
  static constexpr size_t SMEM = (size_t)OFF_BAR + 256 + 1024;  // + alignment slack
  // 4-bit caches: the raw rows of one cache tile, K (codes, then pairs) and V (same) in
  // separate buffers, staged by the producer and dequantized into a K/V stage by warps 10
  // and 11: the copy of the next tile's K overlaps the dequantization of this tile's V
  static constexpr int RAW_CODES = BN * D / 2;
  static constexpr int RAW_HALF = RAW_CODES + BN * 4;
  static constexpr int OFF_RAW = OFF_BAR + 256;
  static constexpr size_t SMEM_KV4 = (size_t)OFF_RAW + 2 * RAW_HALF + 1024;
};

struct Bars {
  uint64_t q_full;
  uint64_t k_full[kNS], k_empty[kNS];
  uint64_t v_full[kNS], v_empty[kNS];
  uint64_t s_full[kQT], p_full[kQT], o_final[kQT];
  uint64_t drain;
  uint32_t tmem_base;
  uint64_t q_free;  // DCA: the MMAs reading the current query vectors have completed
  uint64_t raw_full[2], raw_empty[2];  // 4-bit caches: the staged raw K (0) and V (1) rows of a cache tile
  uint64_t deq_sync;                   // 4-bit caches: both dequantizing warps are done with K or V
};
static_assert(sizeof(Bars) <= 256, "barrier area");

struct Item {
  bool streaming;
  int b, hq, kvh, cidx, qp;  // qp: index of the 256-row block of query rows
};

__device__ __forceinline__ Item item_of(const PrefillParams& p, int idx) {
  Item it;
  const int g = p.sh.g;
  int nk;
  if (idx < p.items_r) {
    it.streaming = false;
    nk = p.sh.n_ret;
  } else {
    idx -= p.items_r;
    it.streaming = true;
    nk = p.sh.n_str;
  }
  const int per_qp = p.sh.B * nk * g;
  if (!it.streaming) {
    // longest query blocks first, in groups of qp_group blocks (about one wave of CTAs
    // per KV head); inside a group, one (sequence, KV head) after the other, so that the
    // CTAs in flight together read the same K/V tiles and each tile comes from DRAM
    // about once (with evict-last loads keeping it in L2 for the CTAs that follow)
    const int GQ = p.qp_group;
    const int grp = idx / (GQ * per_qp);
    const int gs = min(GQ, p.num_qt - grp * GQ);
    int r = idx - grp * GQ * per_qp;
    const int bc = r / (gs * g);
    r %= gs * g;
    it.qp = p.num_qt - 1 - (grp * GQ + r / g);
    it.b = bc / nk;
    it.cidx = bc % nk;
    it.kvh = p.heads.ret_head[it.cidx];
    it.hq = it.kvh * g + (r % g);
    return it;
  }
  const int qp_rev = idx / per_qp;  // longest query blocks first
  int r = idx % per_qp;
  it.qp = p.num_qt - 1 - qp_rev;
  it.b = r / (nk * g);
  r %= nk * g;
  it.cidx = r / g;
  it.kvh = it.streaming ? p.heads.str_head[it.cidx] : p.heads.ret_head[it.cidx];
  it.hq = it.kvh * g + (r % g);
  return it;
}

// The KV tiles a CTA visits: first tiles of the cache (phase 0), then tiles of
// the new tokens (phase 1): [0, sink_eff) for sinks, then [w_lo, k_hi]. Cache tiles
// are [0, n_cache), except for a streaming head kept in a paged pool (rows =
// positions): [0, c_sink) then [c_wlo, c_wlo + n_cache - c_sink).
struct TilePlan {
  int n_cache;
  int c_sink;
  int c_wlo;
  int sink_eff;
  int w_lo;
  int k_hi;
  int total;
};

struct Tile {
  int phase;  // 0 = cache, 1 = new tokens
  int k;      // tile index within its source
};


template <int kMode>
__device__ __forceinline__ TilePlan plan_of(const PrefillParams& p, const Item& it) {
  TilePlan t;
  const int q0 = it.qp * kRows;  // first query row (chunk-local) of the CTA
  const int last_row = min(p.T, q0 + kRows) - 1;
  t.k_hi = last_row / BN;
  if (!it.streaming) {
    t.n_cache = (int)((p.n + BN - 1) / BN);
    t.sink_eff = 0;
    t.w_lo = 0;
  } else if (kMode == kModePool) {
    // sink rows [0, min(S, n)), then the rows the first query row can still see:
    // [max(S, n + q0 - R + 1), n), skipping tiles already taken as sink tiles
    const int64_t sinks = p.sh.S < p.n ? p.sh.S : p.n;
    t.c_sink = (int)((sinks + BN - 1) / BN);
    int64_t w0 = p.n + q0 - p.sh.R + 1;
    if (w0 < p.sh.S) w0 = p.sh.S;
    int wl = (int)(w0 / BN);
    if (wl < t.c_sink) wl = t.c_sink;
    const int te = (int)((p.n + BN - 1) / BN);
    t.c_wlo = wl;
    t.n_cache = t.c_sink + (w0 < p.n && te > wl ? te - wl : 0);
    const int64_t sink_cols = (int64_t)p.sh.S - p.n;  // new tokens that are sinks
    const int sink_tiles = sink_cols > 0 ? (int)((sink_cols + BN - 1) / BN) : 0;
    const int c_lo = q0 - p.sh.R + 1;
    t.w_lo = c_lo > 0 ? c_lo / BN : 0;
    t.sink_eff = sink_tiles < t.w_lo ? sink_tiles : t.w_lo;
    t.total = t.n_cache + t.sink_eff + (t.k_hi - t.w_lo + 1);
    return t;
  } else {
    const int ring_tiles = (p.nvalid + BN - 1) / BN;
    if (q0 + 1 < p.sh.R) {
      t.n_cache = ring_tiles;  // the first rows still see ring entries
    } else {
      const int sinks = p.sh.S < p.nvalid ? p.sh.S : p.nvalid;
      t.n_cache = (sinks + BN - 1) / BN;  // only tiles holding sink slots
    }
    const int64_t sink_cols = (int64_t)p.sh.S - p.n;  // new tokens that are sinks
    const int sink_tiles = sink_cols > 0 ? (int)((sink_cols + BN - 1) / BN) : 0;
    const int c_lo = q0 - p.sh.R + 1;
    t.w_lo = c_lo > 0 ? c_lo / BN : 0;
    t.sink_eff = sink_tiles < t.w_lo ? sink_tiles : t.w_lo;
  }
  t.c_sink = t.n_cache;
  t.c_wlo = 0;
  t.total = t.n_cache + t.sink_eff + (t.k_hi - t.w_lo + 1);
  return t;
}

template <int kMode>
__device__ __forceinline__ Tile tile_at(const TilePlan& pl, int j) {
  Tile t;
  if (j < pl.n_cache) {
    t.phase = 0;
    t.k = (kMode == kModePool && j >= pl.c_sink) ? pl.c_wlo + (j - pl.c_sink) : j;
  } else {
    j -= pl.n_cache;
    t.phase = 1;
    t.k = j < pl.sink_eff ? j : pl.w_lo + (j - pl.sink_eff);
  }
  return t;
}

// Where the cache tiles of one retrieval item lie in a paged pool. Block sizes are
// multiples of 128, so a 128-row tile never crosses a block; everything that does not
// change from tile to tile is worked out once per CTA, leaving one 32-bit division
// per tile on the producer thread.
struct PagedWalk {
  const int32_t* row;  // this item's row of the block table
  int tpb;             // tiles per block
  int last_blk;        // block holding row n - 1 when that block is partly written, else -1
  template <int kMode>
  __device__ __forceinline__ void init(const PrefillParams& p, const Item& it) {
    row = (kMode == kModePool && it.streaming)
              ? p.pg.stream_table + ((int64_t)it.b * p.sh.n_str + it.cidx) * p.pg.max_blocks
              : p.pg.table + ((int64_t)it.b * p.sh.n_ret + it.cidx) * p.pg.max_blocks;
    tpb = p.pg.block_size / BN;
    last_blk = (p.n % p.pg.block_size != 0) ? (int)((p.n - 1) / p.pg.block_size) : -1;
  }
  __device__ __forceinline__ int block_index(int k) const { return (int)((unsigned)k / (unsigned)tpb); }
};

// Dual Chunk Attention: which query vectors (0 query, 1 query_succ, 2 query_inter)
// the 256 query rows of a block use against a key tile. chunk_len and the cache
// length n are multiples of 256, so the block and every tile lie in one chunk each;
// the block's chunk gives two thresholds on the absolute key tile, worked out once
// per CTA. Every head is a retrieval head here, so an item's tiles are the cache
// tiles 0 ... n / 128 - 1 followed by the new-token tiles, and the j-th tile of the
// item is absolute key tile j: the variant needs no tile lookup (the MMA thread
// evaluates it for every tile, on the critical path).
struct DcaTiles {
  int t_intra;  // first key tile of the query block's chunk
  int t_succ;   // first key tile of the chunk before it
  __device__ __forceinline__ void init(const PrefillParams& p, int qp) {
    const int tpc = p.chunk_len / BN;
    // 32-bit: positions stay below 2^31 (checked on the host); a 64-bit division here
    // made the whole DCA prefill 7 % slower
    t_intra = (((int)p.n + qp * kRows) / p.chunk_len) * tpc;
    t_succ = t_intra - tpc;
  }
  __device__ __forceinline__ int var(int j) const { return j >= t_intra ? 0 : (j >= t_succ ? 1 : 2); }
};

__device__ __forceinline__ const CUtensorMap* dca_map(const PrefillParams& p, int v) {
  return v == 0 ? &p.tm_q : (v == 1 ? &p.tm_qs : &p.tm_qi);
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Bits [0, hi) of a 32-bit word (hi clamped to 0 ... 32).
__device__ __forceinline__ uint32_t bits_below(int hi) {
  return hi <= 0 ? 0u : (hi >= 32 ? 0xffffffffu : (1u << hi) - 1u);
}

// Sets masked scores of one 32-column chunk to -inf (columns c0 ... c0+31 of tile t).
// Where the chunk's keys are consecutive positions j0 ... j0+31, the keys row i_abs
// sees form at most two runs (the sinks j < S, and j in (i - R, i]), so the chunk's
// visibility is a 32-bit mask built from a few shifts, applied with one bit test per
// score; ring-cache slots are looked up one by one.
template <int kMode>
__device__ __forceinline__ void mask_chunk(float* v, const PrefillParams& p, const Item& it, const Tile& t, int c0,
                                           int i_abs) {
  const int S = p.sh.S, R = p.sh.R;
  uint32_t vis;
  if (t.phase == 1 || (kMode == kModePool && it.streaming)) {
    // new tokens (j0 = n + tile start), or a streaming head in the pool (row = position)
    const int j0 = t.phase == 1 ? (int)p.n + t.k * BN + c0 : t.k * BN + c0;
    const int d0 = i_abs - j0;  // column e is the key d0 - e positions back
    vis = bits_below(d0 + 1);   // causal: e <= d0
    if (it.streaming) vis &= bits_below(S - j0) | ~bits_below(d0 - R + 1);  // sink, or inside the window
    if (t.phase == 0) vis &= bits_below((int)p.n - j0);                        // rows >= n hold no token
  } else if (!it.streaming) {
    vis = bits_below((int)p.n - t.k * BN - c0);  // rows >= n hold no token
  } else {
    const int32_t* prow = p.pos + (int64_t)it.b * (S + R);
    vis = 0u;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const int slot = t.k * BN + c0 + e;
      const int jp = slot < p.nvalid ? __ldg(prow + slot) : -1;
      vis |= (uint32_t)(jp >= 0 && jp <= i_abs && (jp < S || i_abs - jp < R)) << e;
    }
  }
#pragma unroll
  for (int e = 0; e < 32; ++e)
    if (!((vis >> e) & 1u)) v[e] = -INFINITY;
}

// Row r of a staged 4-bit cache tile into a K or V tile of a stage, laid out as TMA
// writes the bf16 rows (64-column boxes of 128 rows, 128-byte swizzle): value = code *
// scale + zero in fp32, rounded to bf16; a row holding no token is written as zeros. K codes
// are row-major; V codes are in 16-row groups in the decode's fragment order (the byte of
// row k, dims 2 dp and 2 dp + 1, at 4 ((4 (dp / MT) + (k % 8) / 2) MT + dp % MT) + 2 (k % 2)
// + k / 8 of its group, MT = D / 16), so the 4 bytes of dims 8c ... 8c + 7 of a row lie in
// one 16-byte piece, one byte per word.
template <int D, bool kV>
__device__ __forceinline__ void dequant_row(uint8_t* tile, const uint8_t* codes, const uint32_t* sz, int r,
                                            bool valid) {
  constexpr int MT = D / 16;
  float sc = 0.f, zr = 0.f;
  if (valid) {
    const uint32_t w = sz[r];
    sc = __half2float(__ushort_as_half((unsigned short)(w & 0xFFFFu)));
    zr = __half2float(__ushort_as_half((unsigned short)(w >> 16)));
  }
  const int k = r & 15;
  const uint32_t sel = (uint32_t)(2 * (k & 1) + (k >> 3));  // byte of each word (V)
  uint8_t* row = tile + r * 128;
#pragma unroll
  for (int c = 0; c < D / 8; ++c) {  // dims 8c ... 8c + 7: one 16-byte chunk of the row
    uint32_t w = 0;  // byte i: codes of dims 8c + 2i (low nibble), 8c + 2i + 1
    if (valid) {
      if constexpr (kV) {
        const int seg = 4 * ((4 * ((4 * c) / MT) + ((k & 7) >> 1)) * MT + (4 * c) % MT);
        const uint4 q = *reinterpret_cast<const uint4*>(codes + (r & ~15) * (D / 2) + seg);
        w = __byte_perm(__byte_perm(q.x, q.y, sel | ((4u + sel) << 4)), __byte_perm(q.z, q.w, sel | ((4u + sel) << 4)),
                        0x5410);
      } else {
        w = *reinterpret_cast<const uint32_t*>(codes + r * (D / 2) + 4 * c);
      }
    }
    const uint32_t wl = w & 0x0F0F0F0Fu, wh = (w >> 4) & 0x0F0F0F0Fu;
    uint32_t out[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      // a code under the float exponent of 2^23 reads as 2^23 + code; dims 8c + 2i, + 1 as a pair
      float2 c2 = make_float2(__uint_as_float(__byte_perm(wl, 0x4B000000u, 0x7540u | i)),
                              __uint_as_float(__byte_perm(wh, 0x4B000000u, 0x7540u | i)));
      c2 = __fadd2_rn(c2, make_float2(-8388608.f, -8388608.f));
      const float2 val = __ffma2_rn(c2, make_float2(sc, sc), make_float2(zr, zr));
      out[i] = pack_bf16x2(val.x, val.y);
    }
    const int box = c >> 3, cc = c & 7;
    *reinterpret_cast<uint4*>(row + box * kBox + ((cc ^ (r & 7)) << 4)) = make_uint4(out[0], out[1], out[2], out[3]);
  }
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

template <int D, int kMode>
__global__ void __launch_bounds__(Roles<kMode>::kThreads, 1) prefill_kernel(const __grid_constant__ PrefillParams p) {
  using C = PCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  Bars* bars = reinterpret_cast<Bars*>(smem + C::OFF_BAR);

  const DevError err{&g_prefill_err};
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const Item it = item_of(p, blockIdx.x);
  const TilePlan pl = plan_of<kMode>(p, it);
  // After any CTA of this kernel gave up a wait, later CTAs do no work, so a
  // failure ends in about one wait limit instead of one per CTA.
  const int ntiles = (*(volatile unsigned int*)err.word != 0u) ? 0 : pl.total;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < kNS; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    for (int x = 0; x < kQT; ++x) {
      mbar_init(&bars->s_full[x], 1);
      mbar_init(&bars->p_full[x], 4);
      mbar_init(&bars->o_final[x], 1);
    }
    mbar_init(&bars->drain, 1);
    if (kMode == kModeDca) mbar_init(&bars->q_free, 1);
    if (kMode == kModeKv4) {
      for (int h = 0; h < 2; ++h) {
        mbar_init(&bars->raw_full[h], 1);
        mbar_init(&bars->raw_empty[h], 1);
      }
      mbar_init(&bars->deq_sync, Roles<kMode>::kDeqThreads);
    }
    fence_mbarrier_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  if (warp >= 8) {
    // ================================================ warpgroup 2: TMA, MMA, idle
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(Roles<kMode>::kRegsCtl));
    if (warp == kWarpTma) {
      // ------------------------------------------------------------ TMA producer
      if (lane == 0) {
        // DCA: the query vectors of the first key tile; switched when a tile of
        // another chunk relation comes (at most twice per CTA)
        int qvar = 0, q_loads = 1;
        const CUtensorMap* qmap = &p.tm_q;
        DcaTiles dt;
        if (kMode == kModeDca) {
          dt.init(p, it.qp);
          qvar = ntiles > 0 ? dt.var(0) : 0;
          qmap = dca_map(p, qvar);
        }
        prefetch_tmap(qmap);
        // each query tile is read by this CTA alone; K/V tiles by every CTA of the KV head
        const uint64_t pol_kv = l2_policy_evict_last();
        mbar_arrive_expect_tx(&bars->q_full, kQT * C::Q_BYTES);
  #pragma unroll
        for (int x = 0; x < kQT; ++x)
  #pragma unroll
          for (int bx = 0; bx < C::NBOX; ++bx)
            tma_load_4d(sQ + x * C::Q_BYTES + bx * kBox, qmap, bx * 64, it.hq, it.qp * kRows + x * BM, it.b,
                        &bars->q_full);
        bool ok = true;
        // paged: the block id of the next cache tile is read one tile ahead, so its
        // latency overlaps the wait for a free stage
        const bool paged = (kMode == kModePaged && !it.streaming) || kMode == kModePool;
        PagedWalk pw;
        int blk_next = 0;
        if (paged) {
          pw.init<kMode>(p, it);
          if (ntiles > 0 && pl.n_cache > 0)  // (a retrieval item's cache tile 0 is in block 0)
            blk_next = __ldg(pw.row + (kMode == kModePool ? pw.block_index(tile_at<kMode>(pl, 0).k) : 0));
        }
        int j = 0;
        int rc = 0;  // 4-bit caches: raw tiles staged so far
        for (; j < ntiles && ok; ++j) {
          const Tile t = tile_at<kMode>(pl, j);
          if (kMode == kModeDca) {
            const int v = dt.var(j);
            if (v != qvar) {
              // the S MMAs that read the previous query vectors have completed
              if (!mbar_wait(&bars->q_free, (uint32_t)((q_loads - 1) & 1), err, kErrPrefillProducer)) {
                ok = false;
                break;
              }
              qvar = v;
              const CUtensorMap* m = dca_map(p, v);
              mbar_arrive_expect_tx(&bars->q_full, kQT * C::Q_BYTES);
  #pragma unroll
              for (int x = 0; x < kQT; ++x)
  #pragma unroll
                for (int bx = 0; bx < C::NBOX; ++bx)
                  tma_load_4d(sQ + x * C::Q_BYTES + bx * kBox, m, bx * 64, it.hq, it.qp * kRows + x * BM, it.b,
                              &bars->q_full);
              ++q_loads;
            }
          }
          if (kMode == kModeKv4 && t.phase == 0) {
            // a cache tile of 4-bit rows: whole 16-row groups of codes and (scale, zero)
            // pairs into the staging buffer (plane pitches are multiples of 16, so the copy
            // stays in its plane); warps 10 and 11 dequantize them into stage j % kNS and
            // complete its k_full / v_full themselves
            const int64_t r0 = (int64_t)t.k * BN;
            const int64_t keys = it.streaming ? (int64_t)p.nvalid : p.n;
            const int64_t left = (keys - r0 + 15) / 16 * 16;
            const uint32_t rows16 = (uint32_t)(left < BN ? left : BN);
            const int64_t row = (it.streaming ? ((int64_t)it.b * p.sh.n_str + it.cidx) * p.sr16
                                              : ((int64_t)it.b * p.sh.n_ret + it.cidx) * p.cap16) + r0;
            for (int h = 0; h < 2 && ok; ++h) {  // K, then V
              if (!mbar_wait(&bars->raw_empty[h], (uint32_t)((rc & 1) ^ 1), err, kErrPrefillProducer)) {
                ok = false;
                break;
              }
              uint8_t* raw = smem + C::OFF_RAW + h * C::RAW_HALF;
              const uint8_t* codes = h == 0 ? (it.streaming ? p.ks4 : p.k4) : (it.streaming ? p.vs4 : p.v4);
              const uint32_t* pairs = h == 0 ? (it.streaming ? p.kssz : p.ksz) : (it.streaming ? p.vssz : p.vsz);
              mbar_arrive_expect_tx(&bars->raw_full[h], rows16 * (uint32_t)(D / 2 + 4));
              bulk_g2s(raw, codes + row * (D / 2), rows16 * (D / 2), &bars->raw_full[h]);
              bulk_g2s(raw + C::RAW_CODES, pairs + row, rows16 * 4, &bars->raw_full[h]);
            }
            if (!ok) break;
            ++rc;
            continue;
          }
          // paged cache tile: pool block, first row within it, and the maps to read through
          int blk = 0, prow = 0;
          const CUtensorMap* map_k = &p.tm_kfull;
          const CUtensorMap* map_v = &p.tm_vfull;
          if (paged && t.phase == 0) {
            blk = blk_next;
            const int bi = pw.block_index(t.k);
            prow = (t.k - bi * pw.tpb) * BN;
            if (bi == pw.last_blk) {
              map_k = &p.tm_klast;
              map_v = &p.tm_vlast;
            }
            if (j + 1 < pl.n_cache && j + 1 < ntiles)
              blk_next = __ldg(pw.row + pw.block_index(kMode == kModePool ? tile_at<kMode>(pl, j + 1).k : t.k + 1));
            if (blk < 0 || blk >= p.pg.num_blocks) {
              atomicOr(&g_prefill_err, kErrBadBlock);
              blk = p.pg.num_blocks;  // out of range: TMA reads zeros
            }
          }
          const int s = j % kNS;
          const uint32_t ph = (uint32_t)((j / kNS) & 1);
          if (!mbar_wait(&bars->k_empty[s], ph ^ 1u, err, kErrPrefillProducer)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bars->k_full[s], C::KV_BYTES);
          uint8_t* dk = sK + s * C::KV_BYTES;
  #pragma unroll
          for (int bx = 0; bx < C::NBOX; ++bx) {
            if (t.phase == 1)
              tma_load_4d_hint(dk + bx * kBox, &p.tm_k, bx * 64, it.kvh, t.k * BN, it.b, &bars->k_full[s], pol_kv);
            else if (paged)
              tma_load_3d_hint(dk + bx * kBox, map_k, bx * 64, prow, blk, &bars->k_full[s], pol_kv);
            else if (!it.streaming)
              tma_load_3d_hint(dk + bx * kBox, &p.tm_kfull, bx * 64, t.k * BN, it.b * p.sh.n_ret + it.cidx,
                               &bars->k_full[s], pol_kv);
            else
              tma_load_3d_hint(dk + bx * kBox, &p.tm_ksr, bx * 64, t.k * BN, it.b * p.sh.n_str + it.cidx,
                               &bars->k_full[s], pol_kv);
          }
          if (!mbar_wait(&bars->v_empty[s], ph ^ 1u, err, kErrPrefillProducer)) {
            ok = false;
            ++j;  // the K copy of this tile is in flight
            break;
          }
          mbar_arrive_expect_tx(&bars->v_full[s], C::KV_BYTES);
          uint8_t* dv = sV + s * C::KV_BYTES;
  #pragma unroll
          for (int bx = 0; bx < C::NBOX; ++bx) {
            if (t.phase == 1)
              tma_load_4d_hint(dv + bx * kBox, &p.tm_v, bx * 64, it.kvh, t.k * BN, it.b, &bars->v_full[s], pol_kv);
            else if (paged)
              tma_load_3d_hint(dv + bx * kBox, map_v, bx * 64, prow, blk, &bars->v_full[s], pol_kv);
            else if (!it.streaming)
              tma_load_3d_hint(dv + bx * kBox, &p.tm_vfull, bx * 64, t.k * BN, it.b * p.sh.n_ret + it.cidx,
                               &bars->v_full[s], pol_kv);
            else
              tma_load_3d_hint(dv + bx * kBox, &p.tm_vsr, bx * 64, t.k * BN, it.b * p.sh.n_str + it.cidx,
                               &bars->v_full[s], pol_kv);
          }
        }
        if (!ok) {
          // after an early exit, let the copies already issued land before the CTA ends
          mbar_wait(&bars->q_full, kMode == kModeDca ? (uint32_t)((q_loads - 1) & 1) : 0u, err, kErrPrefillProducer);
          for (int jj = (j > kNS ? j - kNS : 0); jj < j; ++jj) {
            if (kMode == kModeKv4 && jj < pl.n_cache) continue;  // filled by the dequantizing warps
            mbar_wait(&bars->k_full[jj % kNS], (uint32_t)((jj / kNS) & 1), err, kErrPrefillProducer);
            mbar_wait(&bars->v_full[jj % kNS], (uint32_t)((jj / kNS) & 1), err, kErrPrefillProducer);
          }
          if (kMode == kModeKv4 && rc > 0)  // the last staging copies
            for (int h = 0; h < 2; ++h) mbar_wait(&bars->raw_full[h], (uint32_t)((rc - 1) & 1), err, kErrPrefillProducer);
        }
      }
    } else if (kMode == kModeKv4 && warp >= kWarpDeq) {
      // ------------------------------------------------------------ 4-bit dequantization
      // The cache tiles come first in an item's tile list; each is staged raw by the
      // producer, and these 192 threads write it into its K/V stage as TMA would have
      // written the bf16 rows (one row of K, then one of V, for each of the first 128),
      // then complete the stage's k_full and v_full.
      const int tid = threadIdx.x - kWarpDeq * 32;
      const int64_t keys = it.streaming ? (int64_t)p.nvalid : p.n;
      bool ok = true;
      for (int j = 0; j < ntiles && j < pl.n_cache && ok; ++j) {
        const Tile t = tile_at<kMode>(pl, j);
        const int s = j % kNS;
        const uint32_t ph = (uint32_t)((j / kNS) & 1);
        const int64_t left = keys - (int64_t)t.k * BN;
        const int rows = left < BN ? (int)left : BN;  // rows of the tile holding a token
        for (int h = 0; h < 2 && ok; ++h) {  // K into sK[s], then V into sV[s]
          const uint8_t* raw = smem + C::OFF_RAW + h * C::RAW_HALF;
          const uint32_t* pairs = reinterpret_cast<const uint32_t*>(raw + C::RAW_CODES);
          if (!mbar_wait(&bars->raw_full[h], (uint32_t)(j & 1), err, kErrPrefillProducer) ||
              !mbar_wait(h == 0 ? &bars->k_empty[s] : &bars->v_empty[s], ph ^ 1u, err, kErrPrefillProducer)) {
            ok = false;
            break;
          }
          uint8_t* tile = (h == 0 ? sK : sV) + s * C::KV_BYTES;
          if (tid < BN) {
            if (h == 0)
              dequant_row<D, false>(tile, raw, pairs, tid, tid < rows);
            else
              dequant_row<D, true>(tile, raw, pairs, tid, tid < rows);
          }
          fence_proxy_async_shared();  // these generic-proxy writes are read by the tensor cores
          mbar_arrive(&bars->deq_sync);
          if (!mbar_wait(&bars->deq_sync, (uint32_t)(h & 1), err, kErrPrefillProducer)) {  // two phases a tile
            ok = false;
            break;
          }
          if (tid == 0) {
            mbar_arrive(h == 0 ? &bars->k_full[s] : &bars->v_full[s]);
            mbar_arrive(&bars->raw_empty[h]);  // the staging buffer may take the next tile's rows
          }
        }
      }
    } else if (warp == kWarpMma) {
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        constexpr uint32_t idesc_s = idesc_bf16_f32(BM, BN, 0, 0);
        constexpr uint32_t idesc_pv = idesc_bf16_f32(BM, D, 0, 1);
        bool ok = mbar_wait(&bars->q_full, 0, err, kErrPrefillMma);
        // Descriptors are built once; a k-step only moves the start address, which
      // lives in the low bits (address >> 4 < 2^14, so the add never carries out).
      const uint64_t dq0 = smem_desc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t dk0 = smem_desc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t dv0 = smem_desc_sw128(smem_u32(sV), kBox, 1024);
      // S_x(jj) = Q_x K(jj)^T
      auto issue_s = [&](int x, int jj) {
        const uint64_t dq = dq0 + (uint64_t)((x * C::Q_BYTES) >> 4);
        const uint64_t dk = dk0 + (uint64_t)(((jj % kNS) * C::KV_BYTES) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = ((kk >> 2) * kBox + (kk & 3) * 32) >> 4;
          mma_ss(tmem + col_s(x), dq + koff, dk + koff, idesc_s, kk > 0 ? 1u : 0u);
        }
        tc_commit(&bars->s_full[x]);
      };
      // O_x += P_x(jj) V(jj)
      auto issue_pv = [&](int x, int jj) {
        const uint64_t dv = dv0 + (uint64_t)(((jj % kNS) * C::KV_BYTES) >> 4);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ts(tmem + col_o(x), tmem + col_s(x) + kk * 8, dv + (uint64_t)((kk * 2048) >> 4), idesc_pv,
                 (jj > 0 || kk > 0) ? 1u : 0u);
      };
      if (ok && ntiles > 0) {
          ok = mbar_wait(&bars->k_full[0], 0, err, kErrPrefillMma);
          if (ok) {
            tc_fence_after();
            issue_s(0, 0);
            issue_s(1, 0);
            tc_commit(&bars->k_empty[0]);
          }
        }
        // DCA: query vectors in shared memory, and the q_full phase of their last load
        DcaTiles dt;
        int qv = 0;
        if (kMode == kModeDca) {
          dt.init(p, it.qp);
          qv = ntiles > 0 ? dt.var(0) : 0;
        }
        uint32_t qph = 0;
        for (int j = 0; j < ntiles && ok; ++j) {
          const int s = j % kNS;
          const bool more = j + 1 < ntiles;
          bool qswitch = false;
          if (kMode == kModeDca && more) {
            const int v = dt.var(j + 1);
            if (v != qv) {
              // S_0(j) and S_1(j), issued before this commit, were the last reads of
              // the current vectors; the producer reloads the buffer once they finish
              qv = v;
              qswitch = true;
              tc_commit(&bars->q_free);
            }
          }
          if (!mbar_wait(&bars->v_full[s], (uint32_t)((j / kNS) & 1), err, kErrPrefillMma)) {
            ok = false;
            break;
          }
          if (more && !mbar_wait(&bars->k_full[(j + 1) % kNS], (uint32_t)(((j + 1) / kNS) & 1), err, kErrPrefillMma)) {
            ok = false;
            break;
          }
          for (int x = 0; x < kQT && ok; ++x) {
            if (!mbar_wait(&bars->p_full[x], (uint32_t)(j & 1), err, kErrPrefillMma)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_pv(x, j);
            if (!more) tc_commit(&bars->o_final[x]);
            if (more) {
              if (kMode == kModeDca && qswitch && x == 0) {
                qph ^= 1u;
                if (!mbar_wait(&bars->q_full, qph, err, kErrPrefillMma)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
              }
              issue_s(x, j + 1);
            }
          }
          if (!ok) break;
          tc_commit(&bars->v_empty[s]);
          if (more) tc_commit(&bars->k_empty[(j + 1) % kNS]);
        }
        // every MMA this thread issued has finished before TMEM is released
        tc_commit(&bars->drain);
        mbar_wait(&bars->drain, 0, err, kErrPrefillMma);
      }
    }
  } else {
    // ================================================ warpgroups 0, 1: softmax
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(Roles<kMode>::kRegsSoftmax));
    const int x = warp >> 2;                     // query tile of this warpgroup
    const int r = (warp & 3) * 32 + lane;        // row within the tile == TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t sbase = lane_base + col_s(x);
    const uint32_t obase = lane_base + col_o(x);
    const int row_local = it.qp * kRows + x * BM + r;  // chunk-local query row
    const int i_abs = (int)p.n + row_local;            // absolute position (< 2^31, checked on the host)
    // DCA: the fp32 per-position scale joins softmax_scale on the fp32 product
    const float sl2 = (kMode == kModeDca && p.mscale && row_local < p.T)
                          ? p.scale_log2 * __ldg(p.mscale + (int64_t)it.b * p.T + row_local)
                          : p.scale_log2;
    const int q_last = x == 0 ? it.qp * kQT : it.qp * kQT + 1;  // diagonal tile of this query tile
    float m_run = -INFINITY;  // running max of scaled scores (log2 units)
    float l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < ntiles && ok; ++j) {
      const Tile t = tile_at<kMode>(pl, j);
      const bool masked = it.streaming || (t.phase == 0 ? (int64_t)(t.k + 1) * BN > p.n : t.k >= q_last);
      if (!mbar_wait(&bars->s_full[x], (uint32_t)(j & 1), err, kErrPrefillSoftmax)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // the whole S row of this thread in one TMEM round trip
      float v[BN];
      {
        uint32_t raw[BN];
        tmem_ld128_sync(sbase, raw);
#pragma unroll
        for (int e = 0; e < BN; ++e) v[e] = __uint_as_float(raw[e]);
      }
      if (masked) {
#pragma unroll
        for (int q4 = 0; q4 < BN / 32; ++q4) mask_chunk<kMode>(v + q4 * 32, p, it, t, q4 * 32, i_abs);
      }
      float mxa = v[0], mxb = v[1];
#pragma unroll
      for (int e = 2; e < BN; e += 4) {
        mxa = max3(mxa, v[e], v[e + 1]);
        if (e + 3 < BN) mxb = max3(mxb, v[e + 2], v[e + 3]);
        else mxb = fmaxf(mxb, v[e + 2]);
      }
      const float mx = fmaxf(mxa, mxb);
      const float mx_s = mx * sl2;
      float f = 1.f;
      if (mx_s > m_run + 8.f) {
        f = ex2_approx(m_run - mx_s);  // 0 while nothing was visible
        l_run *= f;
        m_run = mx_s;
      }
      // O rescale (rare); PV_x(j-1) is complete since S_x(j) is
      if (__any_sync(0xffffffffu, f != 1.f && j > 0)) {
#pragma unroll 1
        for (int q4 = 0; q4 < D / 32; ++q4) {
          uint32_t ov[32];
          tmem_ld32_sync(obase + q4 * 32, ov);
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * f);
          tmem_st32(obase + q4 * 32, ov);
        }
      }
      // P = exp2(s * scale - m), written over the first 64 columns of S
      const float m_use = m_run == -INFINITY ? 0.f : m_run;
      float2 ls = make_float2(0.f, 0.f);
      const float2 sl2x2 = make_float2(sl2, sl2), negm2 = make_float2(-m_use, -m_use);
#pragma unroll
      for (int q4 = 0; q4 < BN / 32; ++q4) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          // s scale - m for a pair of keys in one packed fp32x2 FMA
          const float2 y = __ffma2_rn(make_float2(v[q4 * 32 + 2 * e], v[q4 * 32 + 2 * e + 1]), sl2x2, negm2);
          const float p0 = ex2_approx(y.x);
          const float p1 = ex2_approx(y.y);
          ls = __fadd2_rn(ls, make_float2(p0, p1));
          pk[e] = pack_bf16x2(p0, p1);
        }
        tmem_st16(sbase + q4 * 16, pk);
      }
      l_run += ls.x + ls.y;
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full[x]);
    }
    // ---------------------------------------------------------------- epilogue
    if (ok && ntiles > 0 && mbar_wait(&bars->o_final[x], 0, err, kErrPrefillSoftmax)) {
      tc_fence_after();
      const bool store = row_local < p.T;
      const float inv = 1.f / l_run;
      uint16_t* orow = p.o + (((int64_t)it.b * p.T + row_local) * p.sh.Hq + it.hq) * D;
#pragma unroll 1
      for (int q4 = 0; q4 < D / 32; ++q4) {
        uint32_t ov[32];
        tmem_ld32_sync(obase + q4 * 32, ov);
        if (store) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16x2(__uint_as_float(ov[2 * e]) * inv, __uint_as_float(ov[2 * e + 1]) * inv);
          uint4* dst = reinterpret_cast<uint4*>(orow + q4 * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, int kMode>
cudaError_t launch_t(const PrefillParams& p, cudaStream_t stream) {
  using C = PCfg<D>;
  constexpr size_t smem = kMode == kModeKv4 ? C::SMEM_KV4 : C::SMEM;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(prefill_kernel<D, kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  static int regs = -1;
  if (regs < 0) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, prefill_kernel<D, kMode>);
    if (e != cudaSuccess) return e;
    regs = fa.numRegs;
  }
  // the setmaxnreg split is sized for exactly this launch allocation
  if (regs != Roles<kMode>::kLaunchRegs) return cudaErrorInvalidConfiguration;
  const int grid = p.items_r + p.items_s;
  if (grid == 0) return cudaSuccess;
  prefill_kernel<D, kMode><<<grid, Roles<kMode>::kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

template <int kMode>
cudaError_t launch_mode(const PrefillParams& p, cudaStream_t stream) {
  if (p.sh.D == 128) return launch_t<128, kMode>(p, stream);
  if (p.sh.D == 64) return launch_t<64, kMode>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_prefill(const PrefillParams& p, cudaStream_t stream) {
  if (p.kv4) return launch_mode<kModeKv4>(p, stream);
  if (p.chunk_len > 0) return launch_mode<kModeDca>(p, stream);
  if (p.pg.stream_table) return launch_mode<kModePool>(p, stream);
  return p.pg.table ? launch_mode<kModePaged>(p, stream) : launch_mode<kModePlain>(p, stream);
}

cudaError_t prefill_read_clear_error(uint32_t* code) {
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_prefill_err, sizeof(v));
  if (e != cudaSuccess) return e;
  *code = v;
  if (v) {
    v = 0;
    e = cudaMemcpyToSymbol(g_prefill_err, &v, sizeof(v));
  }
  return e;
}

}  // namespace duo
