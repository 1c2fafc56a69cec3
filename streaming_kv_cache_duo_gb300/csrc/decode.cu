// duo_attn_decode: one query token per sequence against the caches, split over
// the GPU's SMs, merged by log-sum-exp.
//
// Work list. A "unit" is one (sequence, KV head): a retrieval unit holds n keys
// (rows [0, n) of its full cache), a streaming unit min(n, S + R) ring slots.
// Units are cut into tiles of kTK keys and all tiles are laid end to end; CTA c
// takes tiles [c W / C, (c + 1) W / C), so every SM gets the same number of key
// bytes whatever the mix of long retrieval and short streaming units (the
// transformers "Dynamic length in static cache" rule: only the n written
// positions are read, never the capacity).
//
// Per CTA: one producer warp streams the K and V rows of each tile into a
// 4-stage shared-memory ring with 1-D bulk copies (cp.async.bulk, completion on
// an mbarrier); eight consumer warps read each K and V byte once for all g query
// heads of the KV head. Each consumer lane owns 16 (or 8) dims of a key row:
// 128-bit shared loads, fp32 dot products for the g heads, a warp-shuffle
// reduction across the lanes of a key, an online softmax with lazy rescaling
// (the running max moves only when a score exceeds it by 2^8), and fp32
// accumulation of p * v.
//
// Merge. The part of a unit a CTA covers ("segment") ends with a cross-warp merge
// in shared memory. A unit covered by one CTA is written out directly; otherwise
// each segment stores (o, max, sum) in the workspace and the last CTA to arrive
// (atomic ticket, no spinning) merges them:
//     O = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s,
// the merge the vLLM Dual Chunk Attention pull request applies to its partial
// softmax outputs.
#include "duo_device.cuh"

namespace duo {
namespace {

__device__ unsigned int g_decode_err;

constexpr int kTK = kDecodeTK;
constexpr int kStages = 4;
constexpr int kCW = 8;  // consumer warps
constexpr int kThreads = (kCW + 1) * 32;

template <int D, int G>
struct Cfg {
  static constexpr int DPL = (G * 16 <= 64) ? 16 : 8;  // dims per lane
  static constexpr int LPK = D / DPL;                  // lanes per key
  static constexpr int KPI = 32 / LPK;                 // keys per warp iteration
  static constexpr int KPW = kTK / kCW;                // keys per warp per tile
  static constexpr int IT = KPW / KPI;                 // iterations per tile
  static constexpr int CH = DPL / 8;                   // 16-byte chunks per lane
  static constexpr int ROW = D * 2;                    // bytes per key row
  static constexpr int TILE = kTK * ROW;
  static constexpr int STAGE = 2 * TILE;  // K tile, then V tile
  static constexpr int RED = kCW * G * (D + 2);
  static constexpr size_t SMEM = (size_t)kStages * STAGE + (size_t)RED * 4 + 256;
  static_assert(IT >= 1 && KPW % KPI == 0, "tile split");
};

struct Unit {
  int b, kvh;
  bool streaming;
  int64_t keys;
  const uint16_t* kb;
  const uint16_t* vb;
};

__device__ __forceinline__ int64_t unit_start(const DecodeParams& p, int u) {
  return u <= p.U_r ? (int64_t)u * p.tiles_r : (int64_t)p.U_r * p.tiles_r + (int64_t)(u - p.U_r) * p.tiles_s;
}

__device__ __forceinline__ int unit_of(const DecodeParams& p, int64_t t) {
  const int64_t rt = (int64_t)p.U_r * p.tiles_r;
  return t < rt ? (int)(t / p.tiles_r) : p.U_r + (int)((t - rt) / p.tiles_s);
}

// CTA whose tile range contains tile t (ranges are [c W / C, (c + 1) W / C)).
__device__ __forceinline__ int cta_of(const DecodeParams& p, int64_t t) {
  return (int)(((t + 1) * p.C - 1) / p.W);
}

__device__ __forceinline__ Unit unit_info(const DecodeParams& p, int u) {
  Unit x;
  const int D = p.sh.D;
  if (u < p.U_r) {
    const int ri = u % p.sh.n_ret;
    x.b = u / p.sh.n_ret;
    x.kvh = p.heads.ret_head[ri];
    x.streaming = false;
    x.keys = p.n;
    const int64_t off = ((int64_t)x.b * p.sh.n_ret + ri) * p.sh.cap * D;
    x.kb = p.k_full + off;
    x.vb = p.v_full + off;
  } else {
    const int us = u - p.U_r;
    const int si = us % p.sh.n_str;
    x.b = us / p.sh.n_str;
    x.kvh = p.heads.str_head[si];
    x.streaming = true;
    x.keys = p.nvalid;
    const int64_t off = ((int64_t)x.b * p.sh.n_str + si) * (int64_t)(p.sh.S + p.sh.R) * D;
    x.kb = p.k_sr + off;
    x.vb = p.v_sr + off;
  }
  return x;
}

// Synchronisation of the consumer warps through an mbarrier (bounded wait).
struct ConsumerSync {
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

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const DecodeParams p) {
  using C = Cfg<D, G>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stages = smem;
  float* red = reinterpret_cast<float*>(smem + (size_t)kStages * C::STAGE);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)kStages * C::STAGE + (size_t)C::RED * 4);
  uint64_t* empty = full + kStages;
  uint64_t* segbar = empty + kStages;
  int* flag = reinterpret_cast<int*>(segbar + 1);

  const DevError err{&g_decode_err};
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  const int64_t t0 = (int64_t)c * p.W / p.C;
  // After any CTA of this kernel gave up a wait, later CTAs do no work.
  const int64_t t1 = (*(volatile unsigned int*)err.word != 0u) ? t0 : (int64_t)(c + 1) * p.W / p.C;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kCW);
    }
    mbar_init(segbar, kCW);
    fence_mbarrier_init();
  }
  __syncthreads();

  if (warp == kCW) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int64_t j = 0;
      bool ok = true;
      for (int64_t t = t0; t < t1 && ok; ++t, ++j) {
        const int u = unit_of(p, t);
        const Unit x = unit_info(p, u);
        const int64_t lt = t - unit_start(p, u);
        const int64_t rem = x.keys - lt * kTK;
        const int rows = rem < kTK ? (int)rem : kTK;
        const int s = (int)(j % kStages);
        const uint32_t ph = (uint32_t)((j / kStages) & 1);
        if (!mbar_wait(&empty[s], ph ^ 1u, err, kErrDecodeProducer)) {
          ok = false;
          break;
        }
        const uint32_t bytes = (uint32_t)rows * C::ROW;
        mbar_arrive_expect_tx(&full[s], 2 * bytes);
        uint8_t* sk = stages + (size_t)s * C::STAGE;
        bulk_g2s(sk, x.kb + lt * kTK * D, bytes, &full[s]);
        bulk_g2s(sk + C::TILE, x.vb + lt * kTK * D, bytes, &full[s]);
      }
      // Copies still in flight (only after an early exit) land before the CTA ends.
      const int64_t last = j;
      for (int64_t jj = (last > kStages ? last - kStages : 0); jj < last; ++jj)
        mbar_wait(&full[jj % kStages], (uint32_t)((jj / kStages) & 1), err, kErrDecodeProducer);
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int kg = lane / C::LPK;  // key within the warp iteration
    const int cl = lane % C::LPK;  // chunk slot of this lane
    const int SR = p.sh.S + p.sh.R;
    const int64_t pq = p.n - 1;  // query position
    ConsumerSync cs{segbar, 0};
    int64_t j = 0;
    bool ok = true;
    for (int64_t t = t0; t < t1 && ok;) {
      const int u = unit_of(p, t);
      const int64_t us = unit_start(p, u);
      const int64_t ue = unit_start(p, u + 1);
      const int64_t te = ue < t1 ? ue : t1;
      const Unit x = unit_info(p, u);

      // q of the g heads, this lane's dims, pre-scaled by log2(e) / sqrt(D) in fp32.
      float qr[G][C::DPL];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const uint16_t* qh = p.q + ((int64_t)x.b * p.sh.Hq + (int64_t)x.kvh * G + h) * D;
#pragma unroll
        for (int ch = 0; ch < C::CH; ++ch) {
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(qh + (cl + ch * C::LPK) * 8));
          const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            qr[h][ch * 8 + 2 * e] = bf16lo(w4[e]) * p.scale_log2;
            qr[h][ch * 8 + 2 * e + 1] = bf16hi(w4[e]) * p.scale_log2;
          }
        }
      }
      float acc_o[G][C::DPL];
      float l[G], m[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        l[h] = 0.f;
        m[h] = -INFINITY;
#pragma unroll
        for (int e = 0; e < C::DPL; ++e) acc_o[h][e] = 0.f;
      }

      for (; t < te; ++t, ++j) {
        const int s = (int)(j % kStages);
        if (!mbar_wait(&full[s], (uint32_t)((j / kStages) & 1), err, kErrDecodeConsumer)) {
          ok = false;
          break;
        }
        const int64_t lt = t - us;
        const int64_t rem = x.keys - lt * kTK;
        const int rows = rem < kTK ? (int)rem : kTK;
        const uint8_t* sk = stages + (size_t)s * C::STAGE;
        const uint8_t* sv = sk + C::TILE;

        float sc[C::IT][G];
        bool vis[C::IT];
#pragma unroll
        for (int it = 0; it < C::IT; ++it) {
          const int key = warp * C::KPW + it * C::KPI + kg;
          bool valid = key < rows;
          if (x.streaming && valid) {
            const int jp = __ldg(p.pos + (int64_t)x.b * SR + lt * kTK + key);
            valid = jp >= 0 && jp <= pq && (jp < p.sh.S || pq - jp < p.sh.R);
          }
          vis[it] = valid;
          float dot[G];
#pragma unroll
          for (int h = 0; h < G; ++h) dot[h] = 0.f;
#pragma unroll
          for (int ch = 0; ch < C::CH; ++ch) {
            const uint4 kv = *reinterpret_cast<const uint4*>(sk + key * C::ROW + (cl + ch * C::LPK) * 16);
            const uint32_t w4[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float k0 = bf16lo(w4[e]);
              const float k1 = bf16hi(w4[e]);
#pragma unroll
              for (int h = 0; h < G; ++h) {
                dot[h] = fmaf(qr[h][ch * 8 + 2 * e], k0, dot[h]);
                dot[h] = fmaf(qr[h][ch * 8 + 2 * e + 1], k1, dot[h]);
              }
            }
          }
#pragma unroll
          for (int off = 1; off < C::LPK; off <<= 1) {
#pragma unroll
            for (int h = 0; h < G; ++h) dot[h] += __shfl_xor_sync(0xffffffffu, dot[h], off);
          }
#pragma unroll
          for (int h = 0; h < G; ++h) sc[it][h] = valid ? dot[h] : -INFINITY;
        }

        // tile max per head over the warp, lazy rescale of the running state
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float mx = sc[0][h];
#pragma unroll
          for (int it = 1; it < C::IT; ++it) mx = fmaxf(mx, sc[it][h]);
#pragma unroll
          for (int off = C::LPK; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
          if (mx > m[h] + 8.f) {
            const float f = ex2_approx(m[h] - mx);  // 0 when m was -inf
            l[h] *= f;
#pragma unroll
            for (int e = 0; e < C::DPL; ++e) acc_o[h][e] *= f;
            m[h] = mx;
          }
        }
#pragma unroll
        for (int it = 0; it < C::IT; ++it) {
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float pv = vis[it] ? ex2_approx(sc[it][h] - m[h]) : 0.f;
            sc[it][h] = pv;
            l[h] += pv;
          }
        }
#pragma unroll
        for (int it = 0; it < C::IT; ++it) {
          if (vis[it]) {
            const int key = warp * C::KPW + it * C::KPI + kg;
#pragma unroll
            for (int ch = 0; ch < C::CH; ++ch) {
              const uint4 vv = *reinterpret_cast<const uint4*>(sv + key * C::ROW + (cl + ch * C::LPK) * 16);
              const uint32_t w4[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float v0 = bf16lo(w4[e]);
                const float v1 = bf16hi(w4[e]);
#pragma unroll
                for (int h = 0; h < G; ++h) {
                  acc_o[h][ch * 8 + 2 * e] = fmaf(sc[it][h], v0, acc_o[h][ch * 8 + 2 * e]);
                  acc_o[h][ch * 8 + 2 * e + 1] = fmaf(sc[it][h], v1, acc_o[h][ch * 8 + 2 * e + 1]);
                }
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      }
      if (!ok) break;

      // ---------------------------------------------------- segment merge
#pragma unroll
      for (int off = C::LPK; off < 32; off <<= 1) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
          l[h] += __shfl_xor_sync(0xffffffffu, l[h], off);
#pragma unroll
          for (int e = 0; e < C::DPL; ++e) acc_o[h][e] += __shfl_xor_sync(0xffffffffu, acc_o[h][e], off);
        }
      }
      if (kg == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float* r = red + (warp * G + h) * (D + 2);
#pragma unroll
          for (int ch = 0; ch < C::CH; ++ch)
#pragma unroll
            for (int e = 0; e < 8; ++e) r[(cl + ch * C::LPK) * 8 + e] = acc_o[h][ch * 8 + e];
          if (cl == 0) {
            r[D] = m[h];
            r[D + 1] = l[h];
          }
        }
      }
      if (!cs.sync(err)) {
        ok = false;
        break;
      }
      const int tid = threadIdx.x;  // 0 ... 255
      const int c_first = cta_of(p, us);
      const int n_parts = cta_of(p, ue - 1) - c_first + 1;
      float* part = p.partials + (int64_t)(c + u) * G * (D + 2);
      for (int e = tid; e < G * D; e += kCW * 32) {
        const int h = e / D;
        const int d = e % D;
        float M = -INFINITY;
        for (int w = 0; w < kCW; ++w) M = fmaxf(M, red[(w * G + h) * (D + 2) + D]);
        float num = 0.f, den = 0.f;
        for (int w = 0; w < kCW; ++w) {
          const float* r = red + (w * G + h) * (D + 2);
          const float f = r[D] == -INFINITY ? 0.f : ex2_approx(r[D] - M);
          num = fmaf(f, r[d], num);
          den = fmaf(f, r[D + 1], den);
        }
        if (n_parts == 1) {
          p.o[((int64_t)x.b * p.sh.Hq + (int64_t)x.kvh * G + h) * D + d] = __bfloat16_as_ushort(__float2bfloat16_rn(num / den));
        } else {
          part[h * (D + 2) + d] = num;
          if (d == 0) {
            part[h * (D + 2) + D] = M;
            part[h * (D + 2) + D + 1] = den;
          }
        }
      }
      if (n_parts > 1) {
        __threadfence();
        if (!cs.sync(err)) {
          ok = false;
          break;
        }
        if (tid == 0) {
          const unsigned int old = atomicAdd(p.counters + u, 1u);
          const int last = (old == (unsigned int)(n_parts - 1));
          if (last) p.counters[u] = 0u;  // leave the counter at zero for the next call
          *flag = last;
        }
        if (!cs.sync(err)) {
          ok = false;
          break;
        }
        if (*flag) {
          __threadfence();
          for (int e = tid; e < G * D; e += kCW * 32) {
            const int h = e / D;
            const int d = e % D;
            float M = -INFINITY;
            for (int cc = c_first; cc < c_first + n_parts; ++cc)
              M = fmaxf(M, __ldcg(p.partials + ((int64_t)(cc + u) * G + h) * (D + 2) + D));
            float num = 0.f, den = 0.f;
            for (int cc = c_first; cc < c_first + n_parts; ++cc) {
              const float* r = p.partials + ((int64_t)(cc + u) * G + h) * (D + 2);
              const float mm = __ldcg(r + D);
              const float f = mm == -INFINITY ? 0.f : ex2_approx(mm - M);
              num = fmaf(f, __ldcg(r + d), num);
              den = fmaf(f, __ldcg(r + D + 1), den);
            }
            p.o[((int64_t)x.b * p.sh.Hq + (int64_t)x.kvh * G + h) * D + d] = __bfloat16_as_ushort(__float2bfloat16_rn(num / den));
          }
        }
      }
      // the reduction buffer is reused by the next segment
      if (!cs.sync(err)) {
        ok = false;
        break;
      }
    }
  }
  __syncthreads();
}

template <int D, int G>
cudaError_t launch_t(const DecodeParams& p, cudaStream_t stream) {
  using C = Cfg<D, G>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  decode_kernel<D, G><<<p.C, kThreads, C::SMEM, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

size_t decode_workspace_bytes(const Shape& sh, int num_ctas) {
  const int64_t U = (int64_t)sh.B * sh.Hkv;
  const size_t counters = ((size_t)U * 4 + 255) / 256 * 256;
  const size_t parts = (size_t)(num_ctas + U) * sh.g * (sh.D + 2) * 4;
  return counters + parts;
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
