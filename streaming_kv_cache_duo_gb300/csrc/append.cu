// duo_kv_append: write new tokens into the retrieval caches and into the sink +
// ring caches of the streaming heads.
//
// Slot rule (vLLM issue "Could you support Attention Sink?", block tables and
// option 3): token t goes to slot t while t < S and to S + ((t - S) mod R) after
// that; sink slots never move. Of the T tokens of one call only those still held
// when the call ends are written (t < S, or t >= n + T - R), so the result equals
// T single appends and no two threads write the same slot.
//
// Streaming heads kept in a paged pool (block-granular eviction) take every token
// whose block is still live when the call ends instead, at row = position; the host
// passes those tokens as the same two intervals.
//
// HBM-bound copy: one thread moves one 16-byte vector of K and one of V, with
// read-only 128-bit loads from the token-major input and 128-bit stores into the
// head-major caches. Bytes moved: 2 * 2 * D * (T * n_ret + survivors * n_str) per
// sequence, plus 4 bytes of pos per surviving token.
#include <cuda_fp16.h>

#include "duo_device.cuh"

namespace duo {
namespace {

__device__ unsigned int g_append_err;

__global__ void __launch_bounds__(256) append_kernel(const AppendParams p) {
  // a decode launched next may have its CTAs scheduled now (it waits for this grid
  // before it reads anything); this grid, launched as a programmatic dependent itself,
  // writes nothing before the grid before it (a decode reading the ring slots) has ended
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int D = p.sh.D;
  const int Hkv = p.sh.Hkv;
  const int vpr = D / 8;  // 16-byte vectors per row
  const int n_ret = p.sh.n_ret;
  const int n_str = p.sh.n_str;
  const int SR = p.sh.S + p.sh.R;
  const int64_t T = p.T;
  const int64_t ret_vecs = (int64_t)p.sh.B * T * n_ret * vpr;
  const int64_t surv = p.sink_cnt + p.ring_cnt;
  const int64_t str_vecs = (int64_t)p.sh.B * surv * n_str * vpr;
  const int64_t total = ret_vecs + str_vecs;
  const uint4* kin = reinterpret_cast<const uint4*>(p.k_new);
  const uint4* vin = reinterpret_cast<const uint4*>(p.v_new);

  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    if (idx < ret_vecs) {
      int64_t r = idx;
      const int v = (int)(r % vpr);
      r /= vpr;
      const int ri = (int)(r % n_ret);
      r /= n_ret;
      const int64_t t = r % T;
      const int64_t b = r / T;
      const int h = p.heads.ret_head[ri];
      const int64_t src = ((b * T + t) * Hkv + h) * vpr + v;
      const int64_t off = retrieval_row(p.pg, p.sh.cap, D, b * n_ret + ri, p.n + t);
      if (off < 0) {  // paged: block id out of range
        if (v == 0) atomicOr(&g_append_err, kErrBadBlock);
        continue;
      }
      const int64_t dst = off / 8 + v;
      const uint4 kv = __ldg(kin + src);
      const uint4 vv = __ldg(vin + src);
      reinterpret_cast<uint4*>(p.k_full)[dst] = kv;
      reinterpret_cast<uint4*>(p.v_full)[dst] = vv;
    } else {
      int64_t r = idx - ret_vecs;
      const int v = (int)(r % vpr);
      r /= vpr;
      const int si = (int)(r % n_str);
      r /= n_str;
      const int64_t k = r % surv;
      const int64_t b = r / surv;
      const int64_t t_abs = k < p.sink_cnt ? p.sink_lo + k : p.ring_lo + (k - p.sink_cnt);
      const int64_t t = t_abs - p.n;
      const int h = p.heads.str_head[si];
      const int64_t src = ((b * T + t) * Hkv + h) * vpr + v;
      const uint4 kv = __ldg(kin + src);
      const uint4 vv = __ldg(vin + src);
      if (p.pg.stream_table) {  // in the pool, at row = position
        const int64_t off = pool_row(p.pg, p.pg.stream_table, D, b * n_str + si, t_abs);
        if (off < 0) {
          if (v == 0) atomicOr(&g_append_err, kErrBadBlock);
          continue;
        }
        reinterpret_cast<uint4*>(p.k_full)[off / 8 + v] = kv;
        reinterpret_cast<uint4*>(p.v_full)[off / 8 + v] = vv;
        continue;
      }
      const int64_t slot = t_abs < p.sh.S ? t_abs : p.sh.S + (t_abs - p.sh.S) % p.sh.R;
      const int64_t dst = ((b * n_str + si) * SR + slot) * vpr + v;
      reinterpret_cast<uint4*>(p.k_sr)[dst] = kv;
      reinterpret_cast<uint4*>(p.v_sr)[dst] = vv;
      if (si == 0 && v == 0) p.pos[b * SR + slot] = (int32_t)t_abs;
    }
  }
}

// One CTA per sequence: append its one new token at position n_b = seq_lens[b],
// then advance seq_lens[b]. Every thread reads n_b before the barrier and only
// thread 0 writes it after, and no other CTA touches sequence b, so the update
// is race-free. A sequence whose retrieval cache is full is left unchanged and
// the capacity error is recorded.
__global__ void __launch_bounds__(256) append_varlen_kernel(const AppendParams p, int32_t* seq_lens) {
  // a decode launched next may have its CTAs scheduled now (it waits for this grid
  // before it reads anything)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int b = blockIdx.x;
  const int D = p.sh.D;
  const int Hkv = p.sh.Hkv;
  const int vpr = D / 8;
  const int SR = p.sh.S + p.sh.R;
  const int64_t n = seq_lens[b];
  const int64_t cap = p.pg.table ? (int64_t)p.pg.block_size * p.pg.max_blocks : p.sh.cap;
  const bool fits = n >= 0 && (p.sh.n_ret == 0 || n < cap) && n < 0x7fffffff;
  __syncthreads();
  if (fits) {
    const uint4* kin = reinterpret_cast<const uint4*>(p.k_new);
    const uint4* vin = reinterpret_cast<const uint4*>(p.v_new);
    const int64_t slot = n < p.sh.S ? n : p.sh.S + (n - p.sh.S) % p.sh.R;
    for (int idx = threadIdx.x; idx < Hkv * vpr; idx += blockDim.x) {
      const int h = idx / vpr;
      const int v = idx % vpr;
      const int64_t src = ((int64_t)b * Hkv + h) * vpr + v;
      const uint4 kv = __ldg(kin + src);
      const uint4 vv = __ldg(vin + src);
      const int ki = p.heads.kidx[h];
      if (p.heads.kind[h]) {
        const int64_t off = retrieval_row(p.pg, p.sh.cap, D, (int64_t)b * p.sh.n_ret + ki, n);
        if (off < 0) {
          if (v == 0) atomicOr(&g_append_err, kErrBadBlock);
          continue;
        }
        const int64_t dst = off / 8 + v;
        reinterpret_cast<uint4*>(p.k_full)[dst] = kv;
        reinterpret_cast<uint4*>(p.v_full)[dst] = vv;
      } else {
        const int64_t dst = (((int64_t)b * p.sh.n_str + ki) * SR + slot) * vpr + v;
        reinterpret_cast<uint4*>(p.k_sr)[dst] = kv;
        reinterpret_cast<uint4*>(p.v_sr)[dst] = vv;
      }
    }
    if (threadIdx.x == 0 && p.sh.n_str > 0) p.pos[(int64_t)b * SR + slot] = (int32_t)n;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (fits) seq_lens[b] = (int32_t)(n + 1);
    else atomicOr(&g_append_err, kErrAppendCapacity);
  }
}

// 4-bit caches: one warp per (token, head) row of K and V. Each lane holds D / 32
// values of the row; the row's min and max come from warp shuffles, then
//   scale = fp16(fp32((max - min) / 15)),  zero = fp16(min),
//   code  = clamp(rint(fp32(x - zero) / scale), 0, 15)   (0 when scale is 0),
// every step in fp32 round-to-nearest, so the codes are a fixed function of the
// row. Codes are packed two per byte (even dim in the low nibble); lane 0 stores
// the fp16 pair (scale low, zero high). Rows: retrieval rows of all T tokens, then
// the streaming rows the call keeps (the same two intervals as the bf16 ring).
// V codes are stored in the order the decode's tensor-core fragments take them (no
// byte permutes there): within each group of 16 rows, the byte holding the codes of
// row k for dims (2 dp, 2 dp + 1) (low nibble, high nibble) sits at
//     4 ((4 (dp / MT) + ((k & 7) >> 1)) MT + dp % MT) + 2 (k & 1) + (k >> 3),  MT = D / 16,
// so the 32-bit word a lane reads per 16-dim m-tile holds the codes of rows 2t, 2t + 8,
// 2t + 1, 2t + 9 (bytes 0 ... 3) for its two dims. Every byte belongs to one row, so a
// row is written without touching the other rows of its group.
template <int D>
__device__ __forceinline__ int v_code_byte(int k, int dp) {
  constexpr int MT = D / 16;
  return 4 * ((4 * (dp / MT) + ((k & 7) >> 1)) * MT + dp % MT) + 2 * (k & 1) + (k >> 3);
}

// VT = false: `codes` is the row (D / 2 bytes, row-major nibbles); VT = true: `codes` is
// the base of the row's 16-row group and k its row within the group (the V layout).
template <int D, bool VT>
__device__ __forceinline__ void quantize_row(const uint16_t* src, uint8_t* codes, int k, uint32_t* sz, int lane) {
  constexpr int VPL = D / 32;  // values per lane: 4 (D 128) or 2 (D 64)
  float x[VPL];
  if constexpr (VPL == 4) {
    const uint2 w = __ldg(reinterpret_cast<const uint2*>(src) + lane);
    x[0] = bf16lo(w.x);
    x[1] = bf16hi(w.x);
    x[2] = bf16lo(w.y);
    x[3] = bf16hi(w.y);
  } else {
    const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(src) + lane);
    x[0] = bf16lo(w);
    x[1] = bf16hi(w);
  }
  float mn = x[0], mx = x[0];
#pragma unroll
  for (int i = 1; i < VPL; ++i) {
    mn = fminf(mn, x[i]);
    mx = fmaxf(mx, x[i]);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  }
  const __half sh = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), 15.f));
  const __half zh = __float2half_rn(mn);
  const float s = __half2float(sh), z = __half2float(zh);
  uint32_t packed = 0;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    int c = 0;
    if (s != 0.f) {
      c = __float2int_rn(__fdiv_rn(__fsub_rn(x[i], z), s));
      c = c < 0 ? 0 : (c > 15 ? 15 : c);
    }
    packed |= (uint32_t)c << (4 * i);
  }
  if constexpr (VT) {
#pragma unroll
    for (int m = 0; m < VPL / 2; ++m)  // dims (4 lane + 2 m, +1) or (2 lane, +1): pair lane VPL / 2 + m
      codes[v_code_byte<D>(k, lane * (VPL / 2) + m)] = (uint8_t)(packed >> (8 * m));
  } else if constexpr (VPL == 4) {
    reinterpret_cast<uint16_t*>(codes)[lane] = (uint16_t)packed;
  } else {
    codes[lane] = (uint8_t)packed;
  }
  if (lane == 0) *sz = (uint32_t)__half_as_ushort(sh) | ((uint32_t)__half_as_ushort(zh) << 16);
}

template <int D>
__global__ void __launch_bounds__(256) append_kv4_kernel(const AppendParams p) {
  // a decode launched next may have its CTAs scheduled now (it waits for this grid
  // before it reads anything)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int Hkv = p.sh.Hkv;
  const int n_ret = p.sh.n_ret, n_str = p.sh.n_str;
  const int SR = p.sh.S + p.sh.R;
  const int64_t T = p.T;
  const int64_t ret_rows = (int64_t)p.sh.B * T * n_ret;
  const int64_t surv = p.sink_cnt + p.ring_cnt;
  const int64_t total = ret_rows + (int64_t)p.sh.B * surv * n_str;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < total; r += warps) {
    int64_t src_row, dst_row;  // row of [B, T, Hkv] input; row of the destination plane
    bool streaming;
    if (r < ret_rows) {
      const int ri = (int)(r % n_ret);
      const int64_t t = (r / n_ret) % T;
      const int64_t b = r / n_ret / T;
      src_row = (b * T + t) * Hkv + p.heads.ret_head[ri];
      if (p.pg.table) {  // a pool of blocks [num_blocks x block_size rows]
        const int64_t row = p.n + t;
        const int64_t blk = p.pg.table[(b * n_ret + ri) * p.pg.max_blocks + row / p.pg.block_size];
        if (blk < 0 || blk >= p.pg.num_blocks) {
          if (lane == 0) atomicOr(&g_append_err, kErrBadBlock);
          continue;
        }
        dst_row = blk * p.pg.block_size + row % p.pg.block_size;
      } else {
        dst_row = (b * n_ret + ri) * p.cap16 + p.n + t;
      }
      streaming = false;
    } else {
      const int64_t q = r - ret_rows;
      const int si = (int)(q % n_str);
      const int64_t k = (q / n_str) % surv;
      const int64_t b = q / n_str / surv;
      const int64_t t_abs = k < p.sink_cnt ? p.sink_lo + k : p.ring_lo + (k - p.sink_cnt);
      const int64_t slot = t_abs < p.sh.S ? t_abs : p.sh.S + (t_abs - p.sh.S) % p.sh.R;
      src_row = (b * T + (t_abs - p.n)) * Hkv + p.heads.str_head[si];
      dst_row = (b * n_str + si) * p.sr16 + slot;
      streaming = true;
      if (si == 0 && lane == 0) p.pos[b * SR + slot] = (int32_t)t_abs;
    }
    quantize_row<D, false>(p.k_new + src_row * D, (streaming ? p.ks4 : p.k4) + dst_row * (D / 2), 0,
                           (streaming ? p.kssz : p.ksz) + dst_row, lane);
    // plane pitches are multiples of 16 rows, so dst_row's 16-row group starts at dst_row & ~15
    quantize_row<D, true>(p.v_new + src_row * D, (streaming ? p.vs4 : p.v4) + (dst_row & ~int64_t(15)) * (D / 2),
                          (int)(dst_row & 15), (streaming ? p.vssz : p.vsz) + dst_row, lane);
  }
}

}  // namespace

cudaError_t launch_append_kv4(const AppendParams& p, int num_sms, cudaStream_t stream) {
  const int64_t rows = (int64_t)p.sh.B * p.T * p.sh.n_ret + (int64_t)p.sh.B * (p.sink_cnt + p.ring_cnt) * p.sh.n_str;
  if (rows == 0) return cudaSuccess;
  int64_t blocks = (rows + 7) / 8;
  const int64_t cap = (int64_t)num_sms * 8;
  if (blocks > cap) blocks = cap;
  if (p.sh.D == 128)
    append_kv4_kernel<128><<<(unsigned)blocks, 256, 0, stream>>>(p);
  else if (p.sh.D == 64)
    append_kv4_kernel<64><<<(unsigned)blocks, 256, 0, stream>>>(p);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_append_varlen(const AppendParams& p, int32_t* seq_lens, cudaStream_t stream) {
  const int work = p.sh.Hkv * (p.sh.D / 8);
  const int threads = work < 256 ? ((work + 31) / 32) * 32 : 256;
  append_varlen_kernel<<<p.sh.B, threads, 0, stream>>>(p, seq_lens);
  return cudaGetLastError();
}

cudaError_t append_read_clear_error(uint32_t* code) {
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_append_err, sizeof(v));
  if (e != cudaSuccess) return e;
  *code = v;
  if (v) {
    v = 0;
    e = cudaMemcpyToSymbol(g_append_err, &v, sizeof(v));
  }
  return e;
}

cudaError_t launch_append(const AppendParams& p, int num_sms, cudaStream_t stream) {
  const int vpr = p.sh.D / 8;
  const int64_t total = (int64_t)p.sh.B * p.T * p.sh.n_ret * vpr +
                        (int64_t)p.sh.B * (p.sink_cnt + p.ring_cnt) * p.sh.n_str * vpr;
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = (int64_t)num_sms * 8;
  if (blocks > cap) blocks = cap;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, append_kernel, p);
}

}  // namespace duo
