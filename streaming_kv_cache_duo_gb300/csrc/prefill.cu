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
// One CTA computes one 128-row query tile of one query head:
//   warp 4      TMA producer: Q once, then K and V tiles (128 keys x D, 128-byte
//               swizzle) into a 2-stage ring, completion on mbarriers;
//   warp 5      allocates 512 TMEM columns; one thread issues tcgen05.mma:
//               S = Q K^T (A and B from shared memory) into one of two S
//               buffers, and O += P V with P read from TMEM (bf16) and V from
//               shared memory; tcgen05.commit signals each result;
//   warps 0-3   softmax: thread r owns query row r (TMEM lane r): loads its S
//               row with tcgen05.ld, masks it where the tile needs a mask,
//               keeps the running max and sum in fp32 (exp2 with the scale
//               log2(e)/sqrt(D) applied to the fp32 product), rescales O in TMEM
//               only when the max grows by more than 2^8, writes P (bf16) to
//               TMEM; at the end normalises O and stores it.
// S_{j+1} is computed while the softmax works on S_j. Tiles that no row of the
// query tile can see are never visited: a streaming head's query tile visits
// the sink tile(s) and the <= 4 tiles of its window instead of all earlier tiles
// (the block skipping of the block-sparse streaming attention the README uses).
#include "duo_device.cuh"

namespace duo {
namespace {

__device__ unsigned int g_prefill_err;

constexpr int BM = kPrefillBM;
constexpr int BN = kPrefillBN;
constexpr int kNS = 2;  // K/V pipeline stages
constexpr int kWarpTma = 4;
constexpr int kWarpMma = 5;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256, kColP0 = 384, kColP1 = 448;
constexpr int kBox = 128 * 128;  // bytes of a 128-row x 64-column bf16 box

template <int D>
struct PCfg {
  static constexpr int NBOX = D / 64;
  static constexpr int Q_BYTES = BM * D * 2;
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_K + kNS * KV_BYTES;
  static constexpr int OFF_BAR = OFF_V + kNS * KV_BYTES;
  static constexpr size_t SMEM = (size_t)OFF_BAR + 256 + 1024;  // + alignment slack
};

struct Bars {
  uint64_t q_full;
  uint64_t k_full[kNS], k_empty[kNS];
  uint64_t v_full[kNS], v_empty[kNS];
  uint64_t s_full[2], p_full[2], pv_done[2];
  uint64_t drain;
  uint32_t tmem_base;
};

struct Item {
  bool streaming;
  int b, hq, kvh, cidx, qt;
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
  const int per_qt = p.sh.B * nk * g;
  const int qt_rev = idx / per_qt;  // longest query tiles first
  int r = idx % per_qt;
  it.qt = p.num_qt - 1 - qt_rev;
  it.b = r / (nk * g);
  r %= nk * g;
  it.cidx = r / g;
  it.kvh = it.streaming ? p.heads.str_head[it.cidx] : p.heads.ret_head[it.cidx];
  it.hq = it.kvh * g + (r % g);
  return it;
}

// The KV tiles an item visits: first tiles of the cache (phase 0), then tiles of
// the new tokens (phase 1).
struct TilePlan {
  int n_cache;   // cache tiles visited
  int sink_eff;  // new-token tiles [0, sink_eff) for sinks
  int w_lo;      // then new-token tiles [w_lo, qt]
  int total;
};

struct Tile {
  int phase;  // 0 = cache, 1 = new tokens
  int k;      // tile index within its source
  bool masked;
};

__device__ __forceinline__ TilePlan plan_of(const PrefillParams& p, const Item& it) {
  TilePlan t;
  if (!it.streaming) {
    t.n_cache = (int)((p.n + BN - 1) / BN);
    t.sink_eff = 0;
    t.w_lo = 0;
  } else {
    const int ring_tiles = (p.nvalid + BN - 1) / BN;
    if ((int64_t)it.qt * BM + 1 < p.sh.R) {
      t.n_cache = ring_tiles;  // the first rows still see ring entries
    } else {
      const int sinks = p.sh.S < p.nvalid ? p.sh.S : p.nvalid;
      t.n_cache = (sinks + BN - 1) / BN;  // only tiles holding sink slots
    }
    const int64_t sink_cols = (int64_t)p.sh.S - p.n;  // new tokens that are sinks
    const int sink_tiles = sink_cols > 0 ? (int)((sink_cols + BN - 1) / BN) : 0;
    const int64_t c_lo = (int64_t)it.qt * BM - p.sh.R + 1;
    t.w_lo = c_lo > 0 ? (int)(c_lo / BN) : 0;
    t.sink_eff = sink_tiles < t.w_lo ? sink_tiles : t.w_lo;
  }
  t.total = t.n_cache + t.sink_eff + (it.qt - t.w_lo + 1);
  return t;
}

__device__ __forceinline__ Tile tile_at(const PrefillParams& p, const Item& it, const TilePlan& pl, int j) {
  Tile t;
  if (j < pl.n_cache) {
    t.phase = 0;
    t.k = j;
    t.masked = it.streaming || (int64_t)(j + 1) * BN > p.n;
  } else {
    j -= pl.n_cache;
    t.phase = 1;
    t.k = j < pl.sink_eff ? j : pl.w_lo + (j - pl.sink_eff);
    t.masked = it.streaming || t.k == it.qt;
  }
  return t;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ PrefillParams p) {
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
  const TilePlan pl = plan_of(p, it);
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
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->p_full[s], 4);
      mbar_init(&bars->pv_done[s], 1);
    }
    mbar_init(&bars->drain, 1);
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

  if (warp == kWarpTma) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&p.tm_q);
      mbar_arrive_expect_tx(&bars->q_full, C::Q_BYTES);
#pragma unroll
      for (int bx = 0; bx < C::NBOX; ++bx)
        tma_load_4d(sQ + bx * kBox, &p.tm_q, bx * 64, it.hq, it.qt * BM, it.b, &bars->q_full);
      bool ok = true;
      int j = 0;
      for (; j < ntiles && ok; ++j) {
        const Tile t = tile_at(p, it, pl, j);
        const int s = j % kNS;
        const uint32_t ph = (uint32_t)((j / kNS) & 1);
        // K
        if (!mbar_wait(&bars->k_empty[s], ph ^ 1u, err, kErrPrefillProducer)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&bars->k_full[s], C::KV_BYTES);
        uint8_t* dk = sK + s * C::KV_BYTES;
#pragma unroll
        for (int bx = 0; bx < C::NBOX; ++bx) {
          if (t.phase == 1)
            tma_load_4d(dk + bx * kBox, &p.tm_k, bx * 64, it.kvh, t.k * BN, it.b, &bars->k_full[s]);
          else if (!it.streaming)
            tma_load_3d(dk + bx * kBox, &p.tm_kfull, bx * 64, t.k * BN, it.b * p.sh.n_ret + it.cidx, &bars->k_full[s]);
          else
            tma_load_3d(dk + bx * kBox, &p.tm_ksr, bx * 64, t.k * BN, it.b * p.sh.n_str + it.cidx, &bars->k_full[s]);
        }
        // V
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
            tma_load_4d(dv + bx * kBox, &p.tm_v, bx * 64, it.kvh, t.k * BN, it.b, &bars->v_full[s]);
          else if (!it.streaming)
            tma_load_3d(dv + bx * kBox, &p.tm_vfull, bx * 64, t.k * BN, it.b * p.sh.n_ret + it.cidx, &bars->v_full[s]);
          else
            tma_load_3d(dv + bx * kBox, &p.tm_vsr, bx * 64, t.k * BN, it.b * p.sh.n_str + it.cidx, &bars->v_full[s]);
        }
      }
      if (!ok) {
        // after an early exit, let the copies already issued land before the CTA ends
        mbar_wait(&bars->q_full, 0, err, kErrPrefillProducer);
        for (int jj = (j > kNS ? j - kNS : 0); jj < j; ++jj) {
          mbar_wait(&bars->k_full[jj % kNS], (uint32_t)((jj / kNS) & 1), err, kErrPrefillProducer);
          mbar_wait(&bars->v_full[jj % kNS], (uint32_t)((jj / kNS) & 1), err, kErrPrefillProducer);
        }
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(BM, BN, 0, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(BM, D, 0, 1);
      const uint32_t sQa = smem_u32(sQ);
      bool ok = mbar_wait(&bars->q_full, 0, err, kErrPrefillMma);
      auto issue_s = [&](int jj) -> bool {
        const int s = jj % kNS;
        if (!mbar_wait(&bars->k_full[s], (uint32_t)((jj / kNS) & 1), err, kErrPrefillMma)) return false;
        tc_fence_after();
        const uint32_t sKa = smem_u32(sK + s * C::KV_BYTES);
        const uint32_t dS = tmem + ((jj & 1) ? kColS1 : kColS0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * kBox + (kk & 3) * 32;
          mma_ss(dS, smem_desc_sw128(sQa + koff, 16, 1024), smem_desc_sw128(sKa + koff, 16, 1024), idesc_s,
                 kk > 0 ? 1u : 0u);
        }
        tc_commit(&bars->s_full[jj & 1]);
        tc_commit(&bars->k_empty[s]);
        return true;
      };
      if (ok && ntiles > 0) ok = issue_s(0);
      if (ok && ntiles > 1) ok = issue_s(1);
      for (int j = 0; j < ntiles && ok; ++j) {
        const int s = j % kNS;
        if (!mbar_wait(&bars->p_full[j & 1], (uint32_t)((j >> 1) & 1), err, kErrPrefillMma)) {
          ok = false;
          break;
        }
        if (!mbar_wait(&bars->v_full[s], (uint32_t)((j / kNS) & 1), err, kErrPrefillMma)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sVa = smem_u32(sV + s * C::KV_BYTES);
        const uint32_t aP = tmem + ((j & 1) ? kColP1 : kColP0);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          mma_ts(tmem + kColO, aP + kk * 8, smem_desc_sw128(sVa + kk * 2048, kBox, 1024), idesc_pv,
                 (j > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(&bars->pv_done[j & 1]);
        tc_commit(&bars->v_empty[s]);
        if (j + 2 < ntiles) ok = issue_s(j + 2);
      }
      // every MMA this thread issued has finished before TMEM is released
      tc_commit(&bars->drain);
      mbar_wait(&bars->drain, 0, err, kErrPrefillMma);
    }
  } else {
    // ------------------------------------------------------------ softmax (warps 0-3)
    const int r = warp * 32 + lane;  // query row within the tile == TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    const int i_abs = (int)p.n + it.qt * BM + r;  // absolute query position (< 2^31, checked on the host)
    const int S = p.sh.S, R = p.sh.R;
    const float sl2 = p.scale_log2;
    const int SR = S + R;
    float m_run = -INFINITY;  // running max of scaled scores (log2 units)
    float l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < ntiles && ok; ++j) {
      const Tile t = tile_at(p, it, pl, j);
      if (!mbar_wait(&bars->s_full[j & 1], (uint32_t)((j >> 1) & 1), err, kErrPrefillSoftmax)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float sc[BN];
      {
        const uint32_t sbase = lane_base + ((j & 1) ? kColS1 : kColS0);
#pragma unroll
        for (int q4 = 0; q4 < BN / 32; ++q4) {
          uint32_t raw[32];
          tmem_ld32_sync(sbase + q4 * 32, raw);
#pragma unroll
          for (int e = 0; e < 32; ++e) sc[q4 * 32 + e] = __uint_as_float(raw[e]);
        }
      }
      if (t.masked) {
        if (t.phase == 1) {
          // new tokens: key position n + k*BN + c; d = i - j
          const int d0 = i_abs - (p.n + t.k * BN);
#pragma unroll
          for (int c = 0; c < BN; ++c) {
            const int d = d0 - c;
            const int jp = p.n + t.k * BN + c;
            const bool vis = d >= 0 && (!it.streaming || jp < S || d < R);
            if (!vis) sc[c] = -INFINITY;
          }
        } else if (!it.streaming) {
          // retrieval cache: rows >= n hold no token
          const int lim = p.n - t.k * BN;
#pragma unroll
          for (int c = 0; c < BN; ++c)
            if (c >= lim) sc[c] = -INFINITY;
        } else {
          // sink + ring cache: the position of each slot comes from pos[]
          const int32_t* prow = p.pos + (int64_t)it.b * SR;
#pragma unroll
          for (int c = 0; c < BN; ++c) {
            const int slot = t.k * BN + c;
            const int jp = slot < p.nvalid ? __ldg(prow + slot) : -1;
            const bool vis = jp >= 0 && jp <= i_abs && (jp < S || i_abs - jp < R);
            if (!vis) sc[c] = -INFINITY;
          }
        }
      }
      float mx4[4] = {sc[0], sc[1], sc[2], sc[3]};
#pragma unroll
      for (int c = 4; c < BN; ++c) mx4[c & 3] = fmaxf(mx4[c & 3], sc[c]);
      const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
      const float mx_s = mx * sl2;
      float f = 1.f;
      if (mx_s > m_run + 8.f) {
        f = ex2_approx(m_run - mx_s);  // 0 while nothing was visible
        l_run *= f;
        m_run = mx_s;
      }
      // P of tile j overwrites P of tile j - 2: PV(j - 2) must be done
      if (j >= 2 && !mbar_wait(&bars->pv_done[j & 1], (uint32_t)(((j - 2) >> 1) & 1), err, kErrPrefillSoftmax)) {
        ok = false;
        break;
      }
      // O rescale (rare): needs PV(j - 1) done
      if (__any_sync(0xffffffffu, f != 1.f && j > 0)) {
        if (!mbar_wait(&bars->pv_done[(j - 1) & 1], (uint32_t)(((j - 1) >> 1) & 1), err, kErrPrefillSoftmax)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int q4 = 0; q4 < D / 32; ++q4) {
          uint32_t ov[32];
          tmem_ld32_sync(lane_base + kColO + q4 * 32, ov);
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * f);
          tmem_st32(lane_base + kColO + q4 * 32, ov);
        }
        tmem_wait_st();
      }
      const float m_use = m_run == -INFINITY ? 0.f : m_run;
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
      const uint32_t pbase = lane_base + ((j & 1) ? kColP1 : kColP0);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t pk[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float p0 = ex2_approx(fmaf(sc[h * 64 + 2 * e], sl2, -m_use));
          const float p1 = ex2_approx(fmaf(sc[h * 64 + 2 * e + 1], sl2, -m_use));
          ls[e & 3] += p0 + p1;
          pk[e] = pack_bf16x2(p0, p1);
        }
        tmem_st32(pbase + h * 32, pk);
      }
      l_run += (ls[0] + ls[1]) + (ls[2] + ls[3]);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full[j & 1]);
    }
    // ---------------------------------------------------------------- epilogue
    if (ok && ntiles > 0 &&
        mbar_wait(&bars->pv_done[(ntiles - 1) & 1], (uint32_t)(((ntiles - 1) >> 1) & 1), err, kErrPrefillSoftmax)) {
      tc_fence_after();
      const int64_t t_row = (int64_t)it.qt * BM + r;
      const bool store = t_row < p.T;
      const float inv = 1.f / l_run;
      uint16_t* orow = p.o + (((int64_t)it.b * p.T + t_row) * p.sh.Hq + it.hq) * D;
#pragma unroll 1
      for (int q4 = 0; q4 < D / 32; ++q4) {
        uint32_t ov[32];
        tmem_ld32_sync(lane_base + kColO + q4 * 32, ov);
        if (store) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16x2(__uint_as_float(ov[2 * e]) * inv, __uint_as_float(ov[2 * e + 1]) * inv);
          uint4* dst = reinterpret_cast<uint4*>(orow + q4 * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e) dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
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

template <int D>
cudaError_t launch_t(const PrefillParams& p, cudaStream_t stream) {
  using C = PCfg<D>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int grid = p.items_r + p.items_s;
  if (grid == 0) return cudaSuccess;
  prefill_kernel<D><<<grid, kThreads, C::SMEM, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillParams& p, cudaStream_t stream) {
  if (p.sh.D == 128) return launch_t<128>(p, stream);
  if (p.sh.D == 64) return launch_t<64>(p, stream);
  return cudaErrorInvalidValue;
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
