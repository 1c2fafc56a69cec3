// Host side of the C ABI declared in include/duo_attn.h: argument checks, the
// per-head retrieval/streaming map, TMA tensor-map encoding, work sizing and
// kernel dispatch. No device memory is allocated here.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <string>

#include "../../include/duo_attn.h"
#include "duo_internal.h"

using namespace duo;

namespace {

thread_local std::string g_last_error;

duo_status fail(duo_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
duo_status fail(duo_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

duo_status ok() {
  g_last_error.clear();
  return DUO_OK;
}

duo_status cuda_fail(cudaError_t e, const char* what) {
  return fail(DUO_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

}  // namespace

struct duo_handle {
  duo_config cfg;
  Shape sh;
  HeadTable heads;
  int device;
  int num_sms;
  EncodeTiledFn encode;
};

namespace {

// 4-D map over a token-major bf16 tensor [B, T, H, D]; box 64 x 1 x 128 x 1.
duo_status encode_tokens(const duo_handle* h, CUtensorMap* map, const void* base, int B, int T, int H, int D) {
  const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2, (cuuint64_t)T * H * D * 2};
  const cuuint32_t box[4] = {64, 1, (cuuint32_t)kPrefillBM, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = h->encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DUO_ERR_CUDA, "cuTensorMapEncodeTiled (token-major) failed: %d", (int)r);
  return DUO_OK;
}

// 3-D map over a head-major cache [planes, rows_alloc, D] that exposes only the
// first `rows` rows of each plane (later rows read as zero).
duo_status encode_cache(const duo_handle* h, CUtensorMap* map, const void* base, int64_t planes, int64_t rows_alloc,
                        int64_t rows, int D) {
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)rows, (cuuint64_t)planes};
  const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)rows_alloc * D * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)kPrefillBN, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = h->encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DUO_ERR_CUDA, "cuTensorMapEncodeTiled (cache) failed: %d", (int)r);
  return DUO_OK;
}

duo_status check_handle(const duo_handle* h) {
  if (!h) return fail(DUO_ERR_INVALID_ARG, "handle is NULL");
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev != h->device)
    return fail(DUO_ERR_INVALID_ARG, "current device %d differs from the handle's device %d", dev, h->device);
  return DUO_OK;
}

duo_status check_cache(const duo_handle* h, const duo_kv_cache* c, bool need_full, bool need_ring) {
  if (!c) return fail(DUO_ERR_INVALID_ARG, "cache is NULL");
  if (c->n < 0) return fail(DUO_ERR_INVALID_ARG, "cache->n = %lld < 0", (long long)c->n);
  if (need_full && h->sh.n_ret > 0) {
    if (!c->k_full || !c->v_full) return fail(DUO_ERR_INVALID_ARG, "k_full / v_full is NULL");
    if (!aligned16(c->k_full) || !aligned16(c->v_full))
      return fail(DUO_ERR_INVALID_ARG, "k_full / v_full not 16-byte aligned");
  }
  if (need_ring && h->sh.n_str > 0) {
    if (!c->k_sr || !c->v_sr || !c->pos) return fail(DUO_ERR_INVALID_ARG, "k_sr / v_sr / pos is NULL");
    if (!aligned16(c->k_sr) || !aligned16(c->v_sr) || !aligned16(c->pos))
      return fail(DUO_ERR_INVALID_ARG, "k_sr / v_sr / pos not 16-byte aligned");
  }
  return DUO_OK;
}

duo_status check_paged(const duo_handle* h, const duo_paged* pg, PagedLayout* out) {
  *out = PagedLayout{nullptr, 0, 0, 0, nullptr};
  if (!pg) return DUO_OK;
  if (h->sh.n_ret > 0 && (!pg->block_table || (reinterpret_cast<uintptr_t>(pg->block_table) & 3u)))
    return fail(DUO_ERR_INVALID_ARG, "block_table NULL or not 4-byte aligned");
  if (reinterpret_cast<uintptr_t>(pg->stream_table) & 3u)
    return fail(DUO_ERR_INVALID_ARG, "stream_table not 4-byte aligned");
  if (h->sh.n_ret == 0 && !(h->sh.n_str > 0 && pg->stream_table))
    return fail(DUO_ERR_INVALID_ARG, "paged layout with no head in the pool");
  if (pg->block_size < 128 || pg->block_size % 128 != 0)
    return fail(DUO_ERR_UNSUPPORTED, "block_size = %d is not a positive multiple of 128", pg->block_size);
  if (pg->max_blocks < 1 || pg->num_blocks < 1 || pg->num_blocks > 0x7fffffffLL)
    return fail(DUO_ERR_INVALID_ARG, "max_blocks / num_blocks out of range");
  if ((int64_t)pg->block_size * pg->max_blocks > 0x7fffffffLL)
    return fail(DUO_ERR_INVALID_ARG, "block_size x max_blocks >= 2^31");
  *out = PagedLayout{h->sh.n_ret > 0 ? pg->block_table : nullptr, pg->block_size, pg->max_blocks, pg->num_blocks,
                     h->sh.n_str > 0 ? pg->stream_table : nullptr};
  return DUO_OK;
}

bool is_paged(const PagedLayout& pg) { return pg.table || pg.stream_table; }

int64_t retrieval_capacity(const duo_handle* h, const PagedLayout& pg) {
  return is_paged(pg) ? (int64_t)pg.block_size * pg.max_blocks : h->sh.cap;
}

// Tokens a cache can hold: every head kind kept in the pool, or with full rows,
// stops at its capacity; ring caches have none.
duo_status check_capacity(const duo_handle* h, const PagedLayout& pg, int64_t n, duo_status code) {
  const int64_t cap = retrieval_capacity(h, pg);
  const bool bounded = h->sh.n_ret > 0 || pg.stream_table;
  if (bounded && n > cap)
    return fail(code, "%lld tokens exceed the cache capacity %lld", (long long)n, (long long)cap);
  return DUO_OK;
}

// Streaming heads in the pool: logical blocks [lo, hi) hold no token a query at a
// position >= n - 1 can see (past the sink blocks, ending at or before n - R).
void stream_dead_blocks(int64_t S, int64_t R, int64_t bs, int64_t n, int64_t* lo, int64_t* hi) {
  *lo = (S + bs - 1) / bs;
  const int64_t w = n > R ? n - R : 0;
  *hi = w / bs > *lo ? w / bs : *lo;
}

}  // namespace

extern "C" {

const char* duo_last_error(void) { return g_last_error.c_str(); }

const char* duo_status_string(duo_status s) {
  switch (s) {
    case DUO_OK: return "DUO_OK";
    case DUO_ERR_INVALID_ARG: return "DUO_ERR_INVALID_ARG";
    case DUO_ERR_UNSUPPORTED: return "DUO_ERR_UNSUPPORTED";
    case DUO_ERR_CAPACITY: return "DUO_ERR_CAPACITY";
    case DUO_ERR_CUDA: return "DUO_ERR_CUDA";
    case DUO_ERR_DEVICE_TIMEOUT: return "DUO_ERR_DEVICE_TIMEOUT";
    case DUO_ERR_WORKSPACE: return "DUO_ERR_WORKSPACE";
  }
  return "DUO_ERR_UNKNOWN";
}

duo_status duo_classify_heads(const uint8_t* is_retrieval, int32_t num_kv_heads, int32_t* kind_index,
                              int32_t* n_retrieval) {
  if (!is_retrieval || !kind_index || !n_retrieval) return fail(DUO_ERR_INVALID_ARG, "NULL argument");
  if (num_kv_heads < 1 || num_kv_heads > kMaxHeads)
    return fail(DUO_ERR_INVALID_ARG, "num_kv_heads = %d outside [1, %d]", num_kv_heads, kMaxHeads);
  int32_t nr = 0, ns = 0;
  for (int32_t h = 0; h < num_kv_heads; ++h) kind_index[h] = is_retrieval[h] ? nr++ : ns++;
  *n_retrieval = nr;
  return ok();
}

// Head table and shape of a handle for a per-KV-head retrieval mask.
static void set_heads(duo_handle* h, const uint8_t* is_retrieval) {
  const duo_config& c = h->cfg;
  int nr = 0, ns = 0;
  for (int k = 0; k < c.num_kv_heads; ++k) {
    if (is_retrieval[k]) {
      h->heads.ret_head[nr] = (uint8_t)k;
      h->heads.kind[k] = DUO_RETRIEVAL;
      h->heads.kidx[k] = (uint8_t)nr++;
    } else {
      h->heads.str_head[ns] = (uint8_t)k;
      h->heads.kind[k] = DUO_STREAMING;
      h->heads.kidx[k] = (uint8_t)ns++;
    }
  }
  h->sh = Shape{c.batch, c.num_q_heads, c.num_kv_heads, c.head_dim, c.sink_size, c.recent_size,
                c.num_q_heads / c.num_kv_heads, nr, ns, c.max_seq_len};
}

duo_status duo_set_head_mask(duo_handle* h, const uint8_t* is_retrieval) {
  duo_status st = check_handle(h);
  if (st != DUO_OK) return st;
  if (!is_retrieval) return fail(DUO_ERR_INVALID_ARG, "is_retrieval is NULL");
  set_heads(h, is_retrieval);
  return ok();
}

duo_status duo_create(const duo_config* cfg, const uint8_t* is_retrieval, duo_handle** out) {
  if (!cfg || !is_retrieval || !out) return fail(DUO_ERR_INVALID_ARG, "NULL argument");
  *out = nullptr;
  const duo_config& c = *cfg;
  if (c.batch < 1 || c.batch > 65535) return fail(DUO_ERR_INVALID_ARG, "batch = %d outside [1, 65535]", c.batch);
  if (c.num_kv_heads < 1 || c.num_kv_heads > kMaxHeads)
    return fail(DUO_ERR_INVALID_ARG, "num_kv_heads = %d outside [1, %d]", c.num_kv_heads, kMaxHeads);
  if (c.num_q_heads < 1 || c.num_q_heads % c.num_kv_heads != 0)
    return fail(DUO_ERR_INVALID_ARG, "num_q_heads = %d is not a multiple of num_kv_heads = %d", c.num_q_heads,
                c.num_kv_heads);
  const int g = c.num_q_heads / c.num_kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8)
    return fail(DUO_ERR_UNSUPPORTED, "num_q_heads / num_kv_heads = %d not in {1, 2, 4, 8}", g);
  if (c.head_dim != 64 && c.head_dim != 128)
    return fail(DUO_ERR_UNSUPPORTED, "head_dim = %d not in {64, 128}", c.head_dim);
  if (c.sink_size < 0) return fail(DUO_ERR_INVALID_ARG, "sink_size = %d < 0", c.sink_size);
  if (c.recent_size < 1) return fail(DUO_ERR_INVALID_ARG, "recent_size = %d < 1", c.recent_size);
  if ((int64_t)c.sink_size + c.recent_size > (1 << 20))
    return fail(DUO_ERR_UNSUPPORTED, "sink_size + recent_size > 2^20");
  if (c.max_seq_len < 1 || c.max_seq_len > 0x7fffffffLL)
    return fail(DUO_ERR_INVALID_ARG, "max_seq_len = %lld outside [1, 2^31)", (long long)c.max_seq_len);

  duo_handle* h = new (std::nothrow) duo_handle();
  if (!h) return fail(DUO_ERR_INVALID_ARG, "out of host memory");
  h->cfg = c;
  set_heads(h, is_retrieval);

  cudaError_t e = cudaGetDevice(&h->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device);
  int major = 0, minor = 0;
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, h->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, h->device);
  if (e != cudaSuccess) {
    delete h;
    return cuda_fail(e, "device query");
  }
  if (major != 10 || minor != 3) {
    delete h;
    return fail(DUO_ERR_UNSUPPORTED, "device compute capability %d.%d: this library is built for sm_103a only", major,
                minor);
  }
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
    delete h;
    return fail(DUO_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  }
  h->encode = reinterpret_cast<EncodeTiledFn>(fn);
  *out = h;
  return ok();
}

void duo_destroy(duo_handle* h) { delete h; }

duo_status duo_cache_reset(duo_handle* h, duo_kv_cache* c, void* stream) {
  duo_status st = check_handle(h);
  if (st != DUO_OK) return st;
  if (!c) return fail(DUO_ERR_INVALID_ARG, "cache is NULL");
  if (h->sh.n_str > 0) {
    if (!c->pos) return fail(DUO_ERR_INVALID_ARG, "pos is NULL");
    cudaError_t e = cudaMemsetAsync(c->pos, 0xFF, (size_t)h->sh.B * (h->sh.S + h->sh.R) * sizeof(int32_t),
                                    (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(pos)");
  }
  c->n = 0;
  return ok();
}

// 4-bit caches: every array present for the head kinds the handle has, 16-byte
// aligned; the row pitches are the capacities rounded up to 16 rows.
static int64_t pitch16(int64_t rows) { return (rows + 15) / 16 * 16; }

static duo_status check_kv4(const duo_handle* h, const duo_kv_cache* c, const duo_kv4_cache* kv) {
  if (!kv) return fail(DUO_ERR_INVALID_ARG, "kv4 is NULL");
  if (!c) return fail(DUO_ERR_INVALID_ARG, "cache is NULL");
  if (c->n < 0) return fail(DUO_ERR_INVALID_ARG, "cache->n < 0");
  if (h->sh.n_ret > 0) {
    const void* a[] = {kv->k_codes, kv->v_codes, kv->k_sz, kv->v_sz};
    for (const void* x : a)
      if (!x || !aligned16(x)) return fail(DUO_ERR_INVALID_ARG, "retrieval 4-bit arrays NULL or not 16-byte aligned");
  }
  if (h->sh.n_str > 0) {
    const void* a[] = {kv->ks_codes, kv->vs_codes, kv->ks_sz, kv->vs_sz};
    for (const void* x : a)
      if (!x || !aligned16(x)) return fail(DUO_ERR_INVALID_ARG, "streaming 4-bit arrays NULL or not 16-byte aligned");
    if (!c->pos || !aligned16(c->pos)) return fail(DUO_ERR_INVALID_ARG, "pos NULL or not 16-byte aligned");
  }
  return DUO_OK;
}

static duo_status append_impl(duo_handle* h, duo_kv_cache* c, const duo_paged* pgd, const void* k_new,
                              const void* v_new, int32_t T, void* stream, const duo_kv4_cache* kv4 = nullptr) {
  duo_status st = check_handle(h);
  if (st != DUO_OK) return st;
  PagedLayout pg;
  if ((st = check_paged(h, pgd, &pg)) != DUO_OK) return st;
  if (kv4) {
    if ((st = check_kv4(h, c, kv4)) != DUO_OK) return st;
    if (pg.stream_table) return fail(DUO_ERR_UNSUPPORTED, "4-bit caches keep streaming heads in their ring arrays");
  } else if ((st = check_cache(h, c, true, !pg.stream_table)) != DUO_OK) {
    return st;
  }
  if (T < 1) return fail(DUO_ERR_INVALID_ARG, "T = %d < 1", T);
  if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new))
    return fail(DUO_ERR_INVALID_ARG, "k_new / v_new NULL or not 16-byte aligned");
  const Shape& sh = h->sh;
  if (c->n + T > 0x7fffffffLL) return fail(DUO_ERR_CAPACITY, "positions would reach 2^31");
  if ((st = check_capacity(h, pg, c->n + T, DUO_ERR_CAPACITY)) != DUO_OK) return st;
  AppendParams p;
  memset(&p, 0, sizeof(p));
  p.pg = pg;
  p.k_new = static_cast<const uint16_t*>(k_new);
  p.v_new = static_cast<const uint16_t*>(v_new);
  p.k_full = static_cast<uint16_t*>(c->k_full);
  p.v_full = static_cast<uint16_t*>(c->v_full);
  p.k_sr = static_cast<uint16_t*>(c->k_sr);
  p.v_sr = static_cast<uint16_t*>(c->v_sr);
  p.pos = c->pos;
  p.n = c->n;
  p.T = T;
  const int64_t n = c->n, e = c->n + T, S = sh.S, R = sh.R;
  // survivors of the call: t < S, or t >= n + T - R (ring cache); in a pool, every
  // token whose block is still live when the call ends: t < lo * bs or t >= hi * bs
  int64_t sink_end = S, win_lo = e - R;
  if (pg.stream_table) {
    int64_t lo, hi;
    stream_dead_blocks(S, R, pg.block_size, e, &lo, &hi);
    sink_end = lo * pg.block_size;
    win_lo = hi * pg.block_size;
  }
  p.sink_lo = n;
  p.sink_cnt = n < sink_end ? ((e < sink_end ? e : sink_end) - n) : 0;
  int64_t r0 = n;
  if (r0 < sink_end) r0 = sink_end;
  if (r0 < win_lo) r0 = win_lo;
  p.ring_lo = r0;
  p.ring_cnt = e > r0 ? e - r0 : 0;
  p.sh = sh;
  p.heads = h->heads;
  cudaError_t ce;
  if (kv4) {
    p.k4 = static_cast<uint8_t*>(kv4->k_codes);
    p.v4 = static_cast<uint8_t*>(kv4->v_codes);
    p.ks4 = static_cast<uint8_t*>(kv4->ks_codes);
    p.vs4 = static_cast<uint8_t*>(kv4->vs_codes);
    p.ksz = static_cast<uint32_t*>(kv4->k_sz);
    p.vsz = static_cast<uint32_t*>(kv4->v_sz);
    p.kssz = static_cast<uint32_t*>(kv4->ks_sz);
    p.vssz = static_cast<uint32_t*>(kv4->vs_sz);
    p.cap16 = pitch16(sh.cap);
    p.sr16 = (int)pitch16((int64_t)sh.S + sh.R);
    ce = launch_append_kv4(p, h->num_sms, (cudaStream_t)stream);
  } else {
    ce = launch_append(p, h->num_sms, (cudaStream_t)stream);
  }
  if (ce != cudaSuccess) return cuda_fail(ce, "append launch");
  c->n += T;
  return ok();
}

duo_status duo_kv_append(duo_handle* h, duo_kv_cache* c, const void* k_new, const void* v_new, int32_t T,
                         void* stream) {
  return append_impl(h, c, nullptr, k_new, v_new, T, stream);
}

duo_status duo_kv_append_paged(duo_handle* h, duo_kv_cache* c, const duo_paged* paged, const void* k_new,
                               const void* v_new, int32_t T, void* stream) {
  if (!paged) return fail(DUO_ERR_INVALID_ARG, "paged is NULL");
  return append_impl(h, c, paged, k_new, v_new, T, stream);
}

static duo_status prefill_impl(duo_handle* h, const duo_kv_cache* c, const duo_paged* pgd, const void* q,
                               const void* k, const void* v, int32_t T, void* o, int32_t kind_mask, void* stream,
                               const duo_kv4_cache* kv4 = nullptr) {
  duo_status st = check_handle(h);
  if (st != DUO_OK) return st;
  if (!c) return fail(DUO_ERR_INVALID_ARG, "cache is NULL");
  const Shape& sh = h->sh;
  const bool use_cache = c->n > 0;
  PagedLayout pg;
  if ((st = check_paged(h, pgd, &pg)) != DUO_OK) return st;
  if (kv4) {
    if ((st = check_kv4(h, c, kv4)) != DUO_OK) return st;
  } else if ((st = check_cache(h, c, use_cache, use_cache && !pg.stream_table)) != DUO_OK) {
    return st;
  }
  if (T < 1) return fail(DUO_ERR_INVALID_ARG, "T = %d < 1", T);
  if (!q || !k || !v || !o) return fail(DUO_ERR_INVALID_ARG, "q / k / v / o is NULL");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
    return fail(DUO_ERR_INVALID_ARG, "q / k / v / o not 16-byte aligned");
  if (c->n + T > 0x7fffffffLL) return fail(DUO_ERR_INVALID_ARG, "positions would reach 2^31");
  if (kind_mask < 0 || kind_mask > 3) return fail(DUO_ERR_INVALID_ARG, "kind_mask = %d outside [0, 3]", kind_mask);

  PrefillParams p;
  memset(&p, 0, sizeof(p));
  if ((st = encode_tokens(h, &p.tm_q, q, sh.B, T, sh.Hq, sh.D)) != DUO_OK) return st;
  if ((st = encode_tokens(h, &p.tm_k, k, sh.B, T, sh.Hkv, sh.D)) != DUO_OK) return st;
  if ((st = encode_tokens(h, &p.tm_v, v, sh.B, T, sh.Hkv, sh.D)) != DUO_OK) return st;
  const int64_t SR = (int64_t)sh.S + sh.R;
  const int nvalid = (int)(c->n < SR ? c->n : SR);
  if (kv4) {  // cache tiles are dequantized in the kernel; no tensor maps over the caches
    if ((st = check_capacity(h, pg, c->n, DUO_ERR_INVALID_ARG)) != DUO_OK) return st;
    p.k4 = static_cast<const uint8_t*>(kv4->k_codes);
    p.v4 = static_cast<const uint8_t*>(kv4->v_codes);
    p.ks4 = static_cast<const uint8_t*>(kv4->ks_codes);
    p.vs4 = static_cast<const uint8_t*>(kv4->vs_codes);
    p.ksz = static_cast<const uint32_t*>(kv4->k_sz);
    p.vsz = static_cast<const uint32_t*>(kv4->v_sz);
    p.kssz = static_cast<const uint32_t*>(kv4->ks_sz);
    p.vssz = static_cast<const uint32_t*>(kv4->vs_sz);
    p.cap16 = pitch16(sh.cap);
    p.sr16 = (int)pitch16(SR);
    p.kv4 = 1;
  } else if (use_cache && (sh.n_ret > 0 || pg.stream_table)) {
    if ((st = check_capacity(h, pg, c->n, DUO_ERR_INVALID_ARG)) != DUO_OK) return st;
    if (!is_paged(pg)) {
      if ((st = encode_cache(h, &p.tm_kfull, c->k_full, (int64_t)sh.B * sh.n_ret, sh.cap, c->n, sh.D)) != DUO_OK)
        return st;
      if ((st = encode_cache(h, &p.tm_vfull, c->v_full, (int64_t)sh.B * sh.n_ret, sh.cap, c->n, sh.D)) != DUO_OK)
        return st;
    } else {
      // the pool as [num_blocks, block_size, D]; a second view stops at the written rows of the last block
      const int64_t bs = pg.block_size;
      if ((st = encode_cache(h, &p.tm_kfull, c->k_full, pg.num_blocks, bs, bs, sh.D)) != DUO_OK) return st;
      if ((st = encode_cache(h, &p.tm_vfull, c->v_full, pg.num_blocks, bs, bs, sh.D)) != DUO_OK) return st;
      if (c->n % bs) {
        if ((st = encode_cache(h, &p.tm_klast, c->k_full, pg.num_blocks, bs, c->n % bs, sh.D)) != DUO_OK) return st;
        if ((st = encode_cache(h, &p.tm_vlast, c->v_full, pg.num_blocks, bs, c->n % bs, sh.D)) != DUO_OK) return st;
      }
    }
  }
  p.pg = pg;
  if (!kv4 && use_cache && sh.n_str > 0 && !pg.stream_table) {
    if ((st = encode_cache(h, &p.tm_ksr, c->k_sr, (int64_t)sh.B * sh.n_str, SR, nvalid, sh.D)) != DUO_OK) return st;
    if ((st = encode_cache(h, &p.tm_vsr, c->v_sr, (int64_t)sh.B * sh.n_str, SR, nvalid, sh.D)) != DUO_OK) return st;
  }
  p.o = static_cast<uint16_t*>(o);
  p.pos = c->pos;
  p.n = c->n;
  p.T = T;
  p.nvalid = nvalid;
  p.num_qt = (T + kPrefillRowsPerCta - 1) / kPrefillRowsPerCta;
  const int64_t per_kind = (int64_t)sh.B * sh.g * p.num_qt;
  const int64_t ir = (kind_mask & 2) ? per_kind * sh.n_ret : 0;
  const int64_t is = (kind_mask & 1) ? per_kind * sh.n_str : 0;
  if (ir + is > 0x7fffffffLL) return fail(DUO_ERR_UNSUPPORTED, "too many query tiles for one launch");
  p.items_r = (int)ir;
  p.items_s = (int)is;
  // about one wave of CTAs per KV head; at most num_qt, so qp_group x (items per block)
  // stays within the item count (an int)
  p.qp_group = std::max(1, std::min(h->num_sms / sh.g, p.num_qt));
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)sh.D));
  p.sh = sh;
  p.heads = h->heads;
  cudaError_t ce = launch_prefill(p, (cudaStream_t)stream);
  if (ce != cudaSuccess) return cuda_fail(ce, "prefill launch");
  return ok();
}

duo_status duo_attn_prefill(duo_handle* h, const duo_kv_cache* c, const void* q, const void* k, const void* v,
                            int32_t T, void* o, void* stream) {
  return prefill_impl(h, c, nullptr, q, k, v, T, o, 3, stream);
}

duo_status duo_attn_prefill_select(duo_handle* h, const duo_kv_cache* c, const void* q, const void* k,
                                   const void* v, int32_t T, void* o, int32_t kind_mask, void* stream) {
  return prefill_impl(h, c, nullptr, q, k, v, T, o, kind_mask, stream);
}

duo_status duo_attn_prefill_kv4(duo_handle* h, const duo_kv_cache* c, const duo_kv4_cache* kv4, const void* q,
                                const void* k, const void* v, int32_t T, void* o, void* stream) {
  if (!kv4) return fail(DUO_ERR_INVALID_ARG, "kv4 is NULL");
  return prefill_impl(h, c, nullptr, q, k, v, T, o, 3, stream, kv4);
}

duo_status duo_attn_prefill_paged(duo_handle* h, const duo_kv_cache* c, const duo_paged* paged, const void* q,
                                  const void* k, const void* v, int32_t T, void* o, void* stream) {
  if (!paged) return fail(DUO_ERR_INVALID_ARG, "paged is NULL");
  return prefill_impl(h, c, paged, q, k, v, T, o, 3, stream);
}

// tk: keys per tile (kDecodeTK, or kDecodeTKKv4 for 4-bit caches)
static void decode_plan(const duo_handle* h, int64_t n, DecodeParams* p, int ctas_per_sm = 1, int tk = kDecodeTK) {
  const Shape& sh = h->sh;
  p->seq_lens = nullptr;  // uniform length n unless a caller sets device lengths
  p->pg = PagedLayout{nullptr, 0, 0, 0, nullptr};  // contiguous retrieval caches unless paged
  p->s_sink_tiles = p->s_win_lo = 0;
  p->q_succ = p->q_inter = nullptr;  // not Dual Chunk Attention unless a caller sets chunk_len
  p->mscale = nullptr;
  p->chunk_len = 0;
  p->k4 = p->v4 = p->ks4 = p->vs4 = nullptr;  // bf16 caches unless a caller sets 4-bit ones
  p->ksz = p->vsz = p->kssz = p->vssz = nullptr;
  p->cap16 = 0;
  p->sr16 = 0;
  p->kv4 = 0;
  const int64_t SR = (int64_t)sh.S + sh.R;
  p->n = n;
  p->nvalid = (int)(n < SR ? n : SR);
  p->U_r = sh.B * sh.n_ret;
  p->U_s = sh.B * sh.n_str;
  p->tiles_r = (n + tk - 1) / tk;
  p->tiles_s = (p->nvalid + tk - 1) / tk;
  p->W = (int64_t)p->U_r * p->tiles_r;  // retrieval tiles; streaming units are dealt whole
  const int64_t work = p->W + p->U_s;
  const int64_t cmax = (int64_t)h->num_sms * ctas_per_sm;
  p->C = (int)(work < cmax ? work : cmax);
  p->Cr = (int)(p->W < p->C ? p->W : p->C);
  p->s_first = 0;
  if (p->tiles_r <= kDecodeShortTiles && (int64_t)p->U_r + p->U_s <= cmax) {
    // short caches: one CTA per unit, the streaming units on the CTAs after the retrieval
    // ones, so no unit is split and no partial is merged across CTAs (the merge's atomics,
    // fences and reloads cost more than the few tiles a CTA then walks in sequence)
    p->C = p->U_r + p->U_s;
    p->Cr = p->U_r;
    p->s_first = p->U_r;
  }
}

size_t duo_decode_workspace_size(const duo_handle* h, int64_t n) {
  if (!h) return 0;
  DecodeParams p;
  decode_plan(h, n < 1 ? 1 : n, &p);
  (void)p;
  // sized for the largest grid (the 4-bit decode's) so that one workspace serves every n
  return decode_workspace_bytes(h->sh, h->num_sms * kDecodeCtasPerSmKv4);
}

// Dual Chunk Attention arguments of a decode step (nullptr: plain decode).
struct DcaDecode {
  const void* q_succ;
  const void* q_inter;
  const float* mscale;
  int32_t chunk_len;
};

// DCA entry points treat every head as full attention, and need chunk boundaries that
// fall on 256-row blocks / 128-key tiles.
static duo_status check_dca(const duo_handle* h, int32_t chunk_len, const float* mscale) {
  if (h->sh.n_str > 0)
    return fail(DUO_ERR_UNSUPPORTED, "Dual Chunk Attention needs every head to be a retrieval (full) head");
  if (chunk_len < kPrefillRowsPerCta || chunk_len % kPrefillRowsPerCta != 0)
    return fail(DUO_ERR_UNSUPPORTED, "chunk_len = %d is not a positive multiple of %d", chunk_len,
                kPrefillRowsPerCta);
  if (reinterpret_cast<uintptr_t>(mscale) & 3u) return fail(DUO_ERR_INVALID_ARG, "mscale not 4-byte aligned");
  return DUO_OK;
}

static duo_status decode_impl(duo_handle* h, const duo_kv_cache* c, const duo_paged* pgd, const void* q, void* o,
                              void* workspace, size_t ws_bytes, void* stream, const DcaDecode* dca = nullptr,
                              const duo_kv4_cache* kv4 = nullptr) {
  duo_status st = check_handle(h);
  if (st != DUO_OK) return st;
  if (kv4 && (st = check_kv4(h, c, kv4)) != DUO_OK) return st;
  if (kv4 && pgd && pgd->stream_table)
    return fail(DUO_ERR_UNSUPPORTED, "4-bit caches keep streaming heads in their ring arrays");
  if (dca) {
    if ((st = check_dca(h, dca->chunk_len, dca->mscale)) != DUO_OK) return st;
    if (!dca->q_succ || !dca->q_inter || !aligned16(dca->q_succ) || !aligned16(dca->q_inter))
      return fail(DUO_ERR_INVALID_ARG, "q_succ / q_inter NULL or not 16-byte aligned");
  }
  PagedLayout pg;
  if ((st = check_paged(h, pgd, &pg)) != DUO_OK) return st;
  if (!kv4 && (st = check_cache(h, c, true, !pg.stream_table)) != DUO_OK) return st;
  if (c->n < 1) return fail(DUO_ERR_INVALID_ARG, "decode needs the query token appended first (cache->n >= 1)");
  if ((st = check_capacity(h, pg, c->n, DUO_ERR_INVALID_ARG)) != DUO_OK) return st;
  if (!q || !o || !aligned16(q) || !aligned16(o))
    return fail(DUO_ERR_INVALID_ARG, "q / o NULL or not 16-byte aligned");
  const int ctas_per_sm = kv4 ? kDecodeCtasPerSmKv4 : 1;
  const size_t need = decode_workspace_bytes(h->sh, h->num_sms * ctas_per_sm);
  if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(DUO_ERR_INVALID_ARG, "workspace not 256-byte aligned");
  if (!workspace || ws_bytes < need)
    return fail(DUO_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, workspace ? ws_bytes : 0);
  const Shape& sh = h->sh;
  DecodeParams p;
  decode_plan(h, c->n, &p, ctas_per_sm, kv4 ? kDecodeTKKv4 : kDecodeTK);
  p.q = static_cast<const uint16_t*>(q);
  p.o = static_cast<uint16_t*>(o);
  p.k_full = static_cast<const uint16_t*>(c->k_full);
  p.v_full = static_cast<const uint16_t*>(c->v_full);
  p.k_sr = static_cast<const uint16_t*>(c->k_sr);
  p.v_sr = static_cast<const uint16_t*>(c->v_sr);
  p.pos = c->pos;
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)sh.D));
  p.partials = static_cast<float*>(workspace);
  p.sh = sh;
  p.heads = h->heads;
  p.pg = pg;
  if (kv4) {
    p.k4 = static_cast<const uint8_t*>(kv4->k_codes);
    p.v4 = static_cast<const uint8_t*>(kv4->v_codes);
    p.ks4 = static_cast<const uint8_t*>(kv4->ks_codes);
    p.vs4 = static_cast<const uint8_t*>(kv4->vs_codes);
    p.ksz = static_cast<const uint32_t*>(kv4->k_sz);
    p.vsz = static_cast<const uint32_t*>(kv4->v_sz);
    p.kssz = static_cast<const uint32_t*>(kv4->ks_sz);
    p.vssz = static_cast<const uint32_t*>(kv4->vs_sz);
    p.cap16 = pitch16(sh.cap);
    p.sr16 = (int)pitch16((int64_t)sh.S + sh.R);
    p.kv4 = 1;
  }
  if (dca) {
    p.q_succ = static_cast<const uint16_t*>(dca->q_succ);
    p.q_inter = static_cast<const uint16_t*>(dca->q_inter);
    p.mscale = dca->mscale;
    p.chunk_len = dca->chunk_len;
  }
  if (pg.stream_table) {
    // streaming units read rows (= positions) of the pool: the sink tiles, then the
    // tiles of the window [max(S, n - R), n) not already among them
    const int64_t n = c->n;
    const int64_t st_tiles = ((n < sh.S ? n : sh.S) + kDecodeTK - 1) / kDecodeTK;
    const int64_t w0 = n - sh.R > sh.S ? n - sh.R : sh.S;
    int64_t wl = w0 / kDecodeTK;
    if (wl < st_tiles) wl = st_tiles;
    const int64_t te = (n + kDecodeTK - 1) / kDecodeTK;
    p.s_sink_tiles = (int)st_tiles;
    p.s_win_lo = (int)wl;
    p.tiles_s = (int)(st_tiles + (te > wl ? te - wl : 0));
  }
  cudaError_t ce = launch_decode(p, (cudaStream_t)stream);
  if (ce != cudaSuccess) return cuda_fail(ce, "decode launch");
  return ok();
}

duo_status duo_attn_decode(duo_handle* h, const duo_kv_cache* c, const void* q, void* o, void* workspace,
                           size_t ws_bytes, void* stream) {
  return decode_impl(h, c, nullptr, q, o, workspace, ws_bytes, stream);
}

duo_status duo_attn_decode_paged(duo_handle* h, const duo_kv_cache* c, const duo_paged* paged, const void* q,
                                 void* o, void* workspace, size_t ws_bytes, void* stream) {
  if (!paged) return fail(DUO_ERR_INVALID_ARG, "paged is NULL");
  return decode_impl(h, c, paged, q, o, workspace, ws_bytes, stream);
}

duo_status duo_paged_stream_dead_blocks(int32_t sink_size, int32_t recent_size, int32_t block_size, int64_t n,
                                        int64_t* lo, int64_t* hi) {
  if (!lo || !hi) return fail(DUO_ERR_INVALID_ARG, "lo / hi is NULL");
  if (sink_size < 0 || recent_size < 1 || n < 0)
    return fail(DUO_ERR_INVALID_ARG, "sink_size < 0, recent_size < 1 or n < 0");
  if (block_size < 128 || block_size % 128 != 0)
    return fail(DUO_ERR_UNSUPPORTED, "block_size = %d is not a positive multiple of 128", block_size);
  stream_dead_blocks(sink_size, recent_size, block_size, n, lo, hi);
  return ok();
}

duo_status duo_dca_prefill(duo_handle* h, const duo_kv_cache* c, const void* q, const void* q_succ,
                           const void* q_inter, const void* k, const void* v, const float* mscale, int32_t T,
                           int32_t chunk_len, void* o, void* stream) {
  duo_status st = check_handle(h);
  if (st != DUO_OK) return st;
  if ((st = check_dca(h, chunk_len, mscale)) != DUO_OK) return st;
  if (T < 1) return fail(DUO_ERR_INVALID_ARG, "T = %d < 1", T);
  const int64_t n = c ? c->n : 0;
  if (n > 0) {
    if ((st = check_cache(h, c, true, false)) != DUO_OK) return st;
    if (n % kPrefillRowsPerCta != 0)
      return fail(DUO_ERR_UNSUPPORTED, "cache->n = %lld is not a multiple of %d", (long long)n, kPrefillRowsPerCta);
    if (n > h->sh.cap) return fail(DUO_ERR_INVALID_ARG, "cache->n exceeds the retrieval capacity");
  }
  if (n + T > 0x7fffffffLL) return fail(DUO_ERR_INVALID_ARG, "positions would reach 2^31");
  const void* ptrs[] = {q, q_succ, q_inter, k, v, o};
  for (const void* ptr : ptrs)
    if (!ptr || !aligned16(ptr)) return fail(DUO_ERR_INVALID_ARG, "q / q_succ / q_inter / k / v / o NULL or not 16-byte aligned");
  const Shape& sh = h->sh;
  PrefillParams p;
  memset(&p, 0, sizeof(p));
  if ((st = encode_tokens(h, &p.tm_q, q, sh.B, T, sh.Hq, sh.D)) != DUO_OK) return st;
  if ((st = encode_tokens(h, &p.tm_qs, q_succ, sh.B, T, sh.Hq, sh.D)) != DUO_OK) return st;
  if ((st = encode_tokens(h, &p.tm_qi, q_inter, sh.B, T, sh.Hq, sh.D)) != DUO_OK) return st;
  if ((st = encode_tokens(h, &p.tm_k, k, sh.B, T, sh.Hkv, sh.D)) != DUO_OK) return st;
  if ((st = encode_tokens(h, &p.tm_v, v, sh.B, T, sh.Hkv, sh.D)) != DUO_OK) return st;
  if (n > 0) {
    if ((st = encode_cache(h, &p.tm_kfull, c->k_full, (int64_t)sh.B * sh.n_ret, sh.cap, n, sh.D)) != DUO_OK) return st;
    if ((st = encode_cache(h, &p.tm_vfull, c->v_full, (int64_t)sh.B * sh.n_ret, sh.cap, n, sh.D)) != DUO_OK) return st;
  }
  p.o = static_cast<uint16_t*>(o);
  p.n = n;
  p.T = T;
  p.num_qt = (T + kPrefillRowsPerCta - 1) / kPrefillRowsPerCta;
  const int64_t items = (int64_t)sh.B * sh.g * p.num_qt * sh.n_ret;
  if (items > 0x7fffffffLL) return fail(DUO_ERR_UNSUPPORTED, "too many query tiles for one launch");
  p.items_r = (int)items;
  p.items_s = 0;
  p.qp_group = std::max(1, std::min(h->num_sms / sh.g, p.num_qt));
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)sh.D));
  p.sh = sh;
  p.heads = h->heads;
  p.mscale = mscale;
  p.chunk_len = chunk_len;
  cudaError_t ce = launch_prefill(p, (cudaStream_t)stream);
  if (ce != cudaSuccess) return cuda_fail(ce, "DCA prefill launch");
  return ok();
}

duo_status duo_kv_append_kv4(duo_handle* h, duo_kv_cache* c, const duo_kv4_cache* kv4, const void* k_new,
                             const void* v_new, int32_t T, void* stream) {
  if (!kv4) return fail(DUO_ERR_INVALID_ARG, "kv4 is NULL");
  return append_impl(h, c, nullptr, k_new, v_new, T, stream, kv4);
}

duo_status duo_attn_decode_kv4(duo_handle* h, const duo_kv_cache* c, const duo_kv4_cache* kv4, const void* q,
                               void* o, void* workspace, size_t workspace_bytes, void* stream) {
  if (!kv4) return fail(DUO_ERR_INVALID_ARG, "kv4 is NULL");
  return decode_impl(h, c, nullptr, q, o, workspace, workspace_bytes, stream, nullptr, kv4);
}

duo_status duo_kv_append_kv4_paged(duo_handle* h, duo_kv_cache* c, const duo_paged* paged, const duo_kv4_cache* kv4,
                                   const void* k_new, const void* v_new, int32_t T, void* stream) {
  if (!paged) return fail(DUO_ERR_INVALID_ARG, "paged is NULL");
  if (!kv4) return fail(DUO_ERR_INVALID_ARG, "kv4 is NULL");
  return append_impl(h, c, paged, k_new, v_new, T, stream, kv4);
}

duo_status duo_attn_decode_kv4_paged(duo_handle* h, const duo_kv_cache* c, const duo_paged* paged,
                                     const duo_kv4_cache* kv4, const void* q, void* o, void* workspace,
                                     size_t workspace_bytes, void* stream) {
  if (!paged) return fail(DUO_ERR_INVALID_ARG, "paged is NULL");
  if (!kv4) return fail(DUO_ERR_INVALID_ARG, "kv4 is NULL");
  return decode_impl(h, c, paged, q, o, workspace, workspace_bytes, stream, nullptr, kv4);
}

duo_status duo_dca_decode(duo_handle* h, const duo_kv_cache* c, const void* q, const void* q_succ,
                          const void* q_inter, const float* mscale, int32_t chunk_len, void* o, void* workspace,
                          size_t workspace_bytes, void* stream) {
  const DcaDecode dca{q_succ, q_inter, mscale, chunk_len};
  return decode_impl(h, c, nullptr, q, o, workspace, workspace_bytes, stream, &dca);
}

duo_status duo_kv_append_varlen(duo_handle* h, duo_kv_cache* c, int32_t* seq_lens, const void* k_new,
                                const void* v_new, void* stream) {
  duo_status st = check_handle(h);
  if (st != DUO_OK) return st;
  if ((st = check_cache(h, c, true, true)) != DUO_OK) return st;
  if (!seq_lens) return fail(DUO_ERR_INVALID_ARG, "seq_lens is NULL");
  if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new))
    return fail(DUO_ERR_INVALID_ARG, "k_new / v_new NULL or not 16-byte aligned");
  AppendParams p;
  memset(&p, 0, sizeof(p));
  p.k_new = static_cast<const uint16_t*>(k_new);
  p.v_new = static_cast<const uint16_t*>(v_new);
  p.k_full = static_cast<uint16_t*>(c->k_full);
  p.v_full = static_cast<uint16_t*>(c->v_full);
  p.k_sr = static_cast<uint16_t*>(c->k_sr);
  p.v_sr = static_cast<uint16_t*>(c->v_sr);
  p.pos = c->pos;
  p.T = 1;
  p.sh = h->sh;
  p.heads = h->heads;
  cudaError_t ce = launch_append_varlen(p, seq_lens, (cudaStream_t)stream);
  if (ce != cudaSuccess) return cuda_fail(ce, "append (device lengths) launch");
  return ok();
}

duo_status duo_attn_decode_varlen(duo_handle* h, const duo_kv_cache* c, const int32_t* seq_lens, int64_t max_len,
                                  const void* q, void* o, void* workspace, size_t ws_bytes, void* stream) {
  duo_status st = check_handle(h);
  if (st != DUO_OK) return st;
  if ((st = check_cache(h, c, true, true)) != DUO_OK) return st;
  if (!seq_lens) return fail(DUO_ERR_INVALID_ARG, "seq_lens is NULL");
  if (max_len < 1) return fail(DUO_ERR_INVALID_ARG, "max_len = %lld < 1", (long long)max_len);
  if (h->sh.n_ret > 0 && max_len > h->sh.cap) return fail(DUO_ERR_INVALID_ARG, "max_len exceeds max_seq_len");
  if (!q || !o || !aligned16(q) || !aligned16(o))
    return fail(DUO_ERR_INVALID_ARG, "q / o NULL or not 16-byte aligned");
  const size_t need = decode_workspace_bytes(h->sh, h->num_sms);
  if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(DUO_ERR_INVALID_ARG, "workspace not 256-byte aligned");
  if (!workspace || ws_bytes < need)
    return fail(DUO_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, workspace ? ws_bytes : 0);
  const Shape& sh = h->sh;
  DecodeParams p;
  decode_plan(h, max_len, &p);
  p.seq_lens = seq_lens;
  p.q = static_cast<const uint16_t*>(q);
  p.o = static_cast<uint16_t*>(o);
  p.k_full = static_cast<const uint16_t*>(c->k_full);
  p.v_full = static_cast<const uint16_t*>(c->v_full);
  p.k_sr = static_cast<const uint16_t*>(c->k_sr);
  p.v_sr = static_cast<const uint16_t*>(c->v_sr);
  p.pos = c->pos;
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)sh.D));
  p.partials = static_cast<float*>(workspace);
  p.sh = sh;
  p.heads = h->heads;
  cudaError_t ce = launch_decode(p, (cudaStream_t)stream);
  if (ce != cudaSuccess) return cuda_fail(ce, "decode launch (device lengths)");
  return ok();
}

duo_status duo_device_error(uint32_t* code) {
  if (!code) return fail(DUO_ERR_INVALID_ARG, "code is NULL");
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  uint32_t a = 0, b = 0, t = 0, ap = 0;
  if ((e = prefill_read_clear_error(&a)) != cudaSuccess) return cuda_fail(e, "read prefill error word");
  if ((e = decode_read_clear_error(&b)) != cudaSuccess) return cuda_fail(e, "read decode error word");
  if ((e = selftest_read_clear_error(&t)) != cudaSuccess) return cuda_fail(e, "read self-test error word");
  if ((e = append_read_clear_error(&ap)) != cudaSuccess) return cuda_fail(e, "read append error word");
  *code = a | b | t | ap;
  if ((*code & kErrBadBlock) && !(*code & ~(kErrBadBlock | kErrAppendCapacity)))
    return fail(DUO_ERR_INVALID_ARG, "a block table held an id outside [0, num_blocks) (code 0x%x)", *code);
  if (ap && !(a | b | t))
    return fail(DUO_ERR_CAPACITY, "a device-side append found a full retrieval cache (code 0x%x)", *code);
  if (*code) return fail(DUO_ERR_DEVICE_TIMEOUT, "a kernel gave up a bounded wait (code 0x%x)", *code);
  return ok();
}

duo_status duo_selftest_bounded_wait(uint32_t limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 1000000) return fail(DUO_ERR_INVALID_ARG, "limit_us = %u outside [1, 10^6]", limit_us);
  cudaError_t e = launch_selftest_wait((uint64_t)limit_us * 1000u, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  return ok();
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Decode without a caller-provided workspace.
//
// Some callers cannot hand this library device memory for scratch: a serving
// engine that reserved all device memory up front for its own pool, code that
// must not call cudaMalloc/cudaFree because those calls can synchronise the
// device or fragment memory in the middle of a latency-critical loop, or a host
// runtime whose allocator owns every device allocation. For them,
// duo_attn_decode_static() runs the same decode kernel with its scratch (the
// partial softmax results of units split over CTAs) in the array below,
// which belongs to this library's module: every GPU that loads the library keeps
// kStaticScratchBytes of device memory for it until the process exits.
namespace {

constexpr size_t kStaticScratchBytes = (size_t)2 << 20;  // 2 MiB
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_static_scratch_mu;
// Device address of the array per device, and the CUDA context it was looked up in: a
// module loaded into another context (after cudaDeviceReset, or under a context the
// caller made current) may sit at another address, so a new context looks it up again.
struct StaticScratchAddr {
  CUcontext ctx;
  void* ptr;
};
StaticScratchAddr g_static_scratch_addr[kMaxDevices];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

// Looks up the array's device address once per device and context. The name of a
// __device__ variable is only a host-side stand-in; kernels must be given this address.
duo_status static_scratch_address(int device, void** out) {
  if (device < 0 || device >= kMaxDevices) return fail(DUO_ERR_UNSUPPORTED, "device index %d >= %d", device, kMaxDevices);
  static CtxGetCurrentFn get_ctx = nullptr;
  std::lock_guard<std::mutex> lock(g_static_scratch_mu);
  if (!get_ctx) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
      return fail(DUO_ERR_CUDA, "cuCtxGetCurrent entry point unavailable");
    get_ctx = reinterpret_cast<CtxGetCurrentFn>(fn);
  }
  CUcontext ctx = nullptr;
  if (get_ctx(&ctx) != CUDA_SUCCESS || !ctx) return fail(DUO_ERR_CUDA, "no current CUDA context");
  StaticScratchAddr& slot = g_static_scratch_addr[device];
  if (!slot.ptr || slot.ctx != ctx) {
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static decode scratch)");
    if (!ptr) return fail(DUO_ERR_CUDA, "cudaGetSymbolAddress returned NULL for the static decode scratch");
    slot.ctx = ctx;
    slot.ptr = ptr;
  }
  *out = slot.ptr;
  return DUO_OK;
}

}  // namespace

extern "C" duo_status duo_attn_decode_static(duo_handle* h, const duo_kv_cache* c, const void* q, void* o,
                                             void* stream) {
  duo_status st = check_handle(h);
  if (st != DUO_OK) return st;
  if ((st = check_cache(h, c, true, true)) != DUO_OK) return st;
  if (c->n < 1) return fail(DUO_ERR_INVALID_ARG, "decode needs the query token appended first (cache->n >= 1)");
  if (h->sh.n_ret > 0 && c->n > h->sh.cap) return fail(DUO_ERR_INVALID_ARG, "cache->n exceeds max_seq_len");
  if (!q || !o || !aligned16(q) || !aligned16(o))
    return fail(DUO_ERR_INVALID_ARG, "q / o NULL or not 16-byte aligned");
  const size_t need = decode_workspace_bytes(h->sh, h->num_sms);
  if (need > kStaticScratchBytes)
    return fail(DUO_ERR_WORKSPACE,
                "this shape needs %zu bytes of decode scratch, more than the %zu-byte built-in array; "
                "use duo_attn_decode with a caller workspace",
                need, kStaticScratchBytes);
  void* scratch = nullptr;
  if ((st = static_scratch_address(h->device, &scratch)) != DUO_OK) return st;
  const Shape& sh = h->sh;
  DecodeParams p;
  decode_plan(h, c->n, &p);
  p.q = static_cast<const uint16_t*>(q);
  p.o = static_cast<uint16_t*>(o);
  p.k_full = static_cast<const uint16_t*>(c->k_full);
  p.v_full = static_cast<const uint16_t*>(c->v_full);
  p.k_sr = static_cast<const uint16_t*>(c->k_sr);
  p.v_sr = static_cast<const uint16_t*>(c->v_sr);
  p.pos = c->pos;
  p.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)sh.D));
  p.partials = static_cast<float*>(scratch);
  p.sh = sh;
  p.heads = h->heads;
  cudaError_t ce = launch_decode(p, (cudaStream_t)stream);
  if (ce != cudaSuccess) return cuda_fail(ce, "decode launch (static scratch)");
  return ok();
}
