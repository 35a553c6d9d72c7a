// Host side of the C ABI: the layer -> slab map, argument validation, TMA
// descriptor encoding, split-K planning and the launch calls.  No device
// memory is allocated here; every device buffer belongs to the caller.
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <string>

#include "fa_internal.h"

namespace fa {

static thread_local std::string t_msg;

fa_status fail(fa_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_msg = buf;
  return st;
}

static fa_status ok() {
  t_msg.clear();
  return FA_OK;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return 152;   // GB300
  }
  return n;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Slots of the per-device error-word array: each live cache holds one.
static std::mutex g_slot_mu;
static bool g_slot_used[FA_MAX_CACHES];

static int take_err_slot() {
  std::lock_guard<std::mutex> lock(g_slot_mu);
  for (int i = 0; i < FA_MAX_CACHES; ++i)
    if (!g_slot_used[i]) {
      g_slot_used[i] = true;
      return i;
    }
  return -1;
}

static void give_err_slot(int i) {
  if (i < 0 || i >= FA_MAX_CACHES) return;
  std::lock_guard<std::mutex> lock(g_slot_mu);
  g_slot_used[i] = false;
}

// int8 and fp8 slabs: one code byte per element plus an fp32 scale per row
static bool quantised(int kv_dtype) { return kv_dtype != FA_KV_BF16; }
static size_t elem_bytes(int kv_dtype) { return quantised(kv_dtype) ? 1 : 2; }

// ----------------------------------------------------------------- planning
DecodePlan plan_decode(const fa_cache* c, int layer, int B, int max_seq_len, long long max_cta) {
  DecodePlan p;
  const fa_layer_desc& d = c->layers[layer].d;
  const int g = d.num_q_heads / d.num_kv_heads;
  p.head_chunks = (g + 7) / 8;
  if (B <= 0 || max_seq_len <= 0) return p;
  int tiles = (max_seq_len + kTile - 1) / kTile;
  if (d.kind == FA_SLIDING) {
    const int win_tiles = (d.window + kTile - 2) / kTile + 1;   // tiles a W-row window can span
    if (win_tiles < tiles) tiles = win_tiles;
  }
  p.max_tiles = tiles;
  p.units = B * d.num_kv_heads * p.head_chunks;
  // a pipeline step moves 32 KB of K and V; a CTA gets at least 4 steps
  const int tile_bytes = 2 * kTile * d.head_dim * static_cast<int>(elem_bytes(c->kv_dtype));
  p.min_tiles = 4 * (32768 / tile_bytes);
  const long long t_bound = static_cast<long long>(p.units) * tiles;
  const long long slots = max_cta > 0 ? max_cta : 2LL * sm_count();   // two resident CTAs per SM
  long long n = (t_bound + p.min_tiles - 1) / p.min_tiles;
  if (n > slots) n = slots;
  if (n < 1) n = 1;
  p.ncta = static_cast<int>(n);
  if (p.ncta > 1) {
    const size_t rows = static_cast<size_t>(p.ncta + p.units) * 8;   // partial slots x heads
    p.off_ml = (static_cast<size_t>(p.units) * 4 + 255) / 256 * 256;
    p.off_o = p.off_ml + (rows * 2 * sizeof(float) + 255) / 256 * 256;
    p.ws_bytes = p.off_o + rows * d.head_dim * sizeof(float);
  }
  return p;
}

bool pdl_enabled() {
  static int on = -1;
  if (on < 0) {
    const char* e = getenv("FA_PDL");
    on = (e && e[0] == '0') ? 0 : 1;
  }
  return on == 1;
}

// ------------------------------------------------------------ TMA encoding
static PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

// 3-D map over a slab [rows][D]: dim0 = one 128-byte column block, dim1 =
// column block index (stride 128 B), dim2 = row (stride D * elem).  A box of
// (block, 1, 16) lands as 16 rows x 128 B with 128-byte swizzling.
static fa_status encode_slab_map(CUtensorMap* tm, void* base, int D, int kv_dtype, uint64_t rows) {
  auto enc = get_encoder();
  if (!enc) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const uint64_t eb = elem_bytes(kv_dtype);
  const uint64_t blk = 128 / eb;   // elements per 128-byte block
  cuuint64_t dims[3] = {blk, static_cast<cuuint64_t>(D / blk), rows};
  cuuint64_t strides[2] = {128, static_cast<cuuint64_t>(D * eb)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(blk), 1, static_cast<cuuint32_t>(kTile)};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(tm, quantised(kv_dtype) ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                   3, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
  return FA_OK;
}

// The slab again, with the column block as the outermost dimension: dim0 =
// one 128-byte column block, dim1 = row (stride D * elem), dim2 = column
// block (stride 128 B).  A box (block, 16, D / block) is one 16-row tile that
// lands as D / block consecutive 2 KB pieces of 16 rows x 128 B, each
// 128-byte swizzled: the layout of the (block, 1, 16) boxes, in one copy.
static fa_status encode_tile_map(CUtensorMap* tm, void* base, int D, int kv_dtype, uint64_t rows) {
  auto enc = get_encoder();
  if (!enc) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const uint64_t eb = elem_bytes(kv_dtype);
  const uint64_t blk = 128 / eb;
  cuuint64_t dims[3] = {blk, rows, static_cast<cuuint64_t>(D / blk)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D * eb), 128};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(blk), static_cast<cuuint32_t>(kTile), static_cast<cuuint32_t>(D / blk)};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(tm, quantised(kv_dtype) ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                   3, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled (tile map) failed (CUresult %d)", (int)r);
  return FA_OK;
}

// Queries q [N][Hq][D] as 4-D (64-column block elements, head, token, block
// index): a box (64, g, 128/g, 1) lands as 128 rows ordered (token, head) x 128 B.
static fa_status encode_q_map(CUtensorMap* tm, const void* q, int N, int Hq, int D, int g) {
  auto enc = get_encoder();
  if (!enc) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(Hq), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(D / 64)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(Hq) * D * 2, 128};
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(g), static_cast<cuuint32_t>(128 / g), 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(q), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled (q) failed (CUresult %d)", (int)r);
  return FA_OK;
}

// Chunk rows k_ext / v_ext [N][Hkv][D] as 4-D (64 elements, block, KV head,
// token): a box (64, 1, 1, 64) lands as 64 token rows x 128 B.
static fa_status encode_ext_map(CUtensorMap* tm, const void* x, int N, int Hkv, int D) {
  auto enc = get_encoder();
  if (!enc) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(D / 64), static_cast<cuuint64_t>(Hkv), static_cast<cuuint64_t>(N)};
  cuuint64_t strides[3] = {128, static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(Hkv) * D * 2};
  cuuint32_t box[4] = {64, 1, 1, 64};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(x), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled (k/v chunk) failed (CUresult %d)", (int)r);
  return FA_OK;
}

// 2-D map over fp32 scales [rows]: dim0 = 16 scales of one tile, dim1 = tile.
static fa_status encode_scale_map(CUtensorMap* tm, float* base, uint64_t rows) {
  auto enc = get_encoder();
  if (!enc) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(kTile), rows / kTile};
  cuuint64_t strides[1] = {kTile * sizeof(float)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kTile), 1};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled (scales) failed (CUresult %d)", (int)r);
  return FA_OK;
}

cudaError_t set_smem_once(const void* fn, int bytes, unsigned int* done_mask) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned int bit = 1u << (dev & 31);
  if (__atomic_load_n(done_mask, __ATOMIC_ACQUIRE) & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) __atomic_fetch_or(done_mask, bit, __ATOMIC_RELEASE);
  return e;
}

static fa_status check_layer(const fa_cache* c, int32_t layer) {
  if (!c) return fail(FA_ERR_INVALID_ARG, "cache is NULL");
  if (layer < 0 || layer >= static_cast<int32_t>(c->layers.size()))
    return fail(FA_ERR_INVALID_ARG, "layer %d out of range [0, %zu)", layer, c->layers.size());
  return FA_OK;
}

static fa_status check_bound(const fa_cache* c, int32_t layer, const Slab** out) {
  const int o = c->layers[layer].owner;
  const Slab& s = c->slabs[o];
  if (!s.bound) return fail(FA_ERR_NOT_BOUND, "layer %d: slab owner %d has no slab bound", layer, o);
  *out = &s;
  return FA_OK;
}

}  // namespace fa

using namespace fa;

extern "C" {

int32_t fa_version(void) { return 100; }

const char* fa_last_error(void) { return t_msg.c_str(); }

const char* fa_status_string(int32_t st) {
  switch (st) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_NOT_BOUND: return "FA_ERR_NOT_BOUND";
    case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_DEVICE: return "FA_ERR_DEVICE";
    default: return "unknown fa_status";
  }
}

fa_status fa_cache_create(const fa_layer_desc* layers, int32_t n_layers, int32_t num_pages,
                          int32_t page_size, int32_t kv_dtype, fa_cache** out) {
  if (!out) return fail(FA_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!layers || n_layers <= 0) return fail(FA_ERR_INVALID_ARG, "need at least one layer");
  if (num_pages <= 0) return fail(FA_ERR_INVALID_ARG, "num_pages must be positive");
  if (page_size <= 0 || page_size % kTile != 0 || page_size > 256)
    return fail(FA_ERR_UNSUPPORTED, "page_size %d: must be a multiple of %d, at most 256", page_size, kTile);
  if (kv_dtype != FA_KV_BF16 && kv_dtype != FA_KV_INT8 && kv_dtype != FA_KV_FP8)
    return fail(FA_ERR_UNSUPPORTED, "kv_dtype %d unsupported", kv_dtype);
  fa_cache* c = new (std::nothrow) fa_cache();
  if (!c) return fail(FA_ERR_INVALID_ARG, "out of host memory");
  c->err_slot = take_err_slot();
  if (c->err_slot < 0) {
    delete c;
    return fail(FA_ERR_UNSUPPORTED, "at most %d caches may be live at once", FA_MAX_CACHES);
  }
  c->num_pages = num_pages;
  c->page_size = page_size;
  c->kv_dtype = kv_dtype;
  c->layers.resize(n_layers);
  c->slabs.resize(n_layers);
  for (int i = 0; i < n_layers; ++i) {
    const fa_layer_desc& d = layers[i];
    Layer& L = c->layers[i];
    L.d = d;
    fa_status st = FA_OK;
    if (d.kind != FA_FULL && d.kind != FA_SLIDING)
      st = fail(FA_ERR_INVALID_ARG, "layer %d: kind %d", i, d.kind);
    else if (d.head_dim != 256 && d.head_dim != 512)
      st = fail(FA_ERR_UNSUPPORTED, "layer %d: head_dim %d (supported: 256, 512)", i, d.head_dim);
    else if (d.num_kv_heads <= 0 || d.num_q_heads <= 0 || d.num_q_heads % d.num_kv_heads != 0)
      st = fail(FA_ERR_INVALID_ARG, "layer %d: Hq %d must be a positive multiple of Hkv %d", i,
                d.num_q_heads, d.num_kv_heads);
    else if (d.kind == FA_SLIDING && d.window < 1)
      st = fail(FA_ERR_INVALID_ARG, "layer %d: sliding window %d must be >= 1", i, d.window);
    else if (!(d.sm_scale > 0.0f) || d.sm_scale > 1e30f)
      st = fail(FA_ERR_INVALID_ARG, "layer %d: sm_scale must be positive and finite", i);
    else if (static_cast<int64_t>(num_pages) * d.num_kv_heads * page_size >= (1LL << 31))
      st = fail(FA_ERR_UNSUPPORTED, "layer %d: num_pages * Hkv * page_size must stay below 2^31", i);
    if (st != FA_OK) {
      fa_cache_destroy(c);
      return st;
    }
    if (d.kv_source == FA_KV_OWN) {
      L.owner = i;
      continue;
    }
    // source rule: the last earlier owning layer of the same kind
    int last = -1;
    for (int j = 0; j < i; ++j)
      if (c->layers[j].owner == j && c->layers[j].d.kind == d.kind) last = j;
    int src = d.kv_source == FA_KV_AUTO ? last : d.kv_source;
    if (last < 0) st = fail(FA_ERR_UNSUPPORTED, "layer %d: KV-shared layer with no earlier owning layer of its kind", i);
    else if (d.kv_source != FA_KV_AUTO &&
             (src < 0 || src >= i || c->layers[src].owner != src || c->layers[src].d.kind != d.kind))
      st = fail(FA_ERR_UNSUPPORTED, "layer %d: source %d is not an earlier owning layer of its kind", i, src);
    else if (c->layers[src].d.head_dim != d.head_dim || c->layers[src].d.num_kv_heads != d.num_kv_heads)
      st = fail(FA_ERR_UNSUPPORTED, "layer %d: KV geometry differs from its source %d", i, src);
    if (st != FA_OK) {
      fa_cache_destroy(c);
      return st;
    }
    L.owner = src;
  }
  *out = c;
  return ok();
}

void fa_cache_destroy(fa_cache* c) {
  if (!c) return;
  give_err_slot(c->err_slot);
  delete c;
}

fa_status fa_cache_set_flags(fa_cache* c, uint32_t flags) {
  if (!c) return fail(FA_ERR_INVALID_ARG, "cache is NULL");
  if (flags & ~static_cast<uint32_t>(FA_FLAG_EARLY_METADATA | FA_FLAG_EXTEND_SPLIT_ALL))
    return fail(FA_ERR_INVALID_ARG, "unknown flags 0x%x", flags);
  c->flags = flags;
  return ok();
}

fa_status fa_cache_set_window_pool(fa_cache* c, int32_t window_pages) {
  if (!c) return fail(FA_ERR_INVALID_ARG, "cache is NULL");
  if (window_pages < 0) return fail(FA_ERR_INVALID_ARG, "window_pages must be >= 0");
  for (size_t i = 0; i < c->layers.size(); ++i) {
    const Layer& L = c->layers[i];
    if (L.d.kind != FA_SLIDING) continue;
    if (c->slabs[i].bound) return fail(FA_ERR_INVALID_ARG, "set the window pool before binding sliding slabs (layer %zu is bound)", i);
    const int64_t pages = window_pages > 0 ? window_pages : c->num_pages;
    if (pages * L.d.num_kv_heads * c->page_size >= (1LL << 31))
      return fail(FA_ERR_UNSUPPORTED, "layer %zu: window_pages * Hkv * page_size must stay below 2^31", i);
  }
  c->window_pages = window_pages;
  return ok();
}

fa_status fa_cache_layer_source(const fa_cache* c, int32_t layer, int32_t* slab_owner) {
  fa_status st = check_layer(c, layer);
  if (st) return st;
  if (!slab_owner) return fail(FA_ERR_INVALID_ARG, "slab_owner is NULL");
  *slab_owner = c->layers[layer].owner;
  return ok();
}

fa_status fa_cache_slab_bytes(const fa_cache* c, int32_t layer, size_t* kv_bytes, size_t* scale_bytes) {
  fa_status st = check_layer(c, layer);
  if (st) return st;
  if (!kv_bytes || !scale_bytes) return fail(FA_ERR_INVALID_ARG, "output pointer is NULL");
  const Layer& L = c->layers[layer];
  if (L.owner != layer) {
    *kv_bytes = *scale_bytes = 0;
    return ok();
  }
  const size_t rows = static_cast<size_t>(layer_pages(c, layer)) * L.d.num_kv_heads * c->page_size;
  *kv_bytes = rows * L.d.head_dim * elem_bytes(c->kv_dtype);
  *scale_bytes = quantised(c->kv_dtype) ? rows * sizeof(float) : 0;
  return ok();
}

fa_status fa_cache_bind_slab(fa_cache* c, int32_t layer, void* k, void* v, float* k_scale, float* v_scale) {
  fa_status st = check_layer(c, layer);
  if (st) return st;
  const Layer& L = c->layers[layer];
  if (L.owner != layer)
    return fail(FA_ERR_INVALID_ARG, "layer %d is KV-shared (reads layer %d's slab); bind the source", layer,
                L.owner);
  if (!k || !v) return fail(FA_ERR_INVALID_ARG, "layer %d: k and v must be non-NULL", layer);
  if (!aligned16(k) || !aligned16(v)) return fail(FA_ERR_INVALID_ARG, "layer %d: k, v must be 16-byte aligned", layer);
  if (quantised(c->kv_dtype)) {
    if (!k_scale || !v_scale) return fail(FA_ERR_INVALID_ARG, "layer %d: the 8-bit formats need k_scale and v_scale", layer);
    if (!aligned16(k_scale) || !aligned16(v_scale))
      return fail(FA_ERR_INVALID_ARG, "layer %d: scales must be 16-byte aligned", layer);
  }
  Slab& s = c->slabs[layer];
  const uint64_t rows = static_cast<uint64_t>(layer_pages(c, layer)) * L.d.num_kv_heads * c->page_size;
  st = encode_slab_map(&s.tm_k, k, L.d.head_dim, c->kv_dtype, rows);
  if (st) return st;
  st = encode_slab_map(&s.tm_v, v, L.d.head_dim, c->kv_dtype, rows);
  if (st) return st;
  if ((st = encode_tile_map(&s.tm_kt, k, L.d.head_dim, c->kv_dtype, rows))) return st;
  if ((st = encode_tile_map(&s.tm_vt, v, L.d.head_dim, c->kv_dtype, rows))) return st;
  if (quantised(c->kv_dtype)) {
    if ((st = encode_scale_map(&s.tm_ks, k_scale, rows))) return st;
    if ((st = encode_scale_map(&s.tm_vs, v_scale, rows))) return st;
  } else {
    s.tm_ks = s.tm_k;   // unused in bf16; keeps the kernel parameters defined
    s.tm_vs = s.tm_v;
  }
  // the error word this cache's kernels report into starts clean on this
  // device (its slot may have served a cache destroyed earlier)
  cudaError_t ce = clear_device_error_word(c);
  if (ce != cudaSuccess) return fail(FA_ERR_CUDA, "clearing the device error word: %s", cudaGetErrorString(ce));
  s.k = k;
  s.v = v;
  s.k_scale = quantised(c->kv_dtype) ? k_scale : nullptr;
  s.v_scale = quantised(c->kv_dtype) ? v_scale : nullptr;
  s.bound = true;
  return ok();
}

size_t fa_kv_bytes_per_token(const fa_cache* c, int32_t kind) {
  if (!c) return 0;
  size_t total = 0;
  for (size_t i = 0; i < c->layers.size(); ++i) {
    const Layer& L = c->layers[i];
    if (L.owner != static_cast<int>(i) || L.d.kind != kind) continue;
    const size_t row = quantised(c->kv_dtype) ? L.d.head_dim + sizeof(float) : 2 * L.d.head_dim;
    total += 2 * L.d.num_kv_heads * row;
  }
  return total;
}

fa_status fa_kv_store(fa_cache* c, int32_t layer, const void* k, const void* v, const int32_t* slot_mapping,
                      int32_t T, void* stream) {
  fa_status st = check_layer(c, layer);
  if (st) return st;
  const Layer& L = c->layers[layer];
  if (L.owner != layer) return ok();   // a shared layer stores nothing
  if (T < 0) return fail(FA_ERR_INVALID_ARG, "T must be >= 0");
  if (T == 0) return ok();
  const Slab* s = nullptr;
  if ((st = check_bound(c, layer, &s))) return st;
  if (!k || !v || !slot_mapping) return fail(FA_ERR_INVALID_ARG, "k, v, slot_mapping must be non-NULL");
  if (!aligned16(k) || !aligned16(v)) return fail(FA_ERR_INVALID_ARG, "k, v must be 16-byte aligned");
  cudaError_t ce;
  unsigned int* err = device_error_word(c, &ce);
  if (!err) return fail(FA_ERR_CUDA, "device error word: %s", cudaGetErrorString(ce));
  StoreArgs a{k, v, slot_mapping, s->k, s->v, s->k_scale, s->v_scale, T, L.d.num_kv_heads, L.d.head_dim,
              c->page_size, layer_pages(c, layer), c->kv_dtype, (c->flags & FA_FLAG_EARLY_METADATA) ? 1 : 0, err};
  ce = launch_store(a, static_cast<cudaStream_t>(stream));
  if (ce != cudaSuccess) return fail(FA_ERR_CUDA, "store launch: %s", cudaGetErrorString(ce));
  return ok();
}

size_t fa_decode_workspace_bytes(const fa_cache* c, int32_t layer, int32_t B, int32_t max_seq_len) {
  if (check_layer(c, layer) != FA_OK || B <= 0 || max_seq_len <= 0) return 0;
  return plan_decode(c, layer, B, max_seq_len).ws_bytes;
}

fa_status fa_kv_store_layers(fa_cache* c, int32_t n, const int32_t* layers, const void* const* k,
                             const void* const* v, const int32_t* const* slot_mapping, int32_t T, void* stream) {
  if (!c) return fail(FA_ERR_INVALID_ARG, "cache is NULL");
  if (n < 1 || n > FA_MAX_LAYERS_PER_LAUNCH) return fail(FA_ERR_INVALID_ARG, "n must be in [1, %d]", FA_MAX_LAYERS_PER_LAUNCH);
  if (!layers || !k || !v || !slot_mapping) return fail(FA_ERR_INVALID_ARG, "layers, k, v, slot_mapping must be non-NULL");
  if (T < 0) return fail(FA_ERR_INVALID_ARG, "T must be >= 0");
  fa_status st;
  StoreArgs a[FA_MAX_LAYERS_PER_LAUNCH];
  int m = 0;
  cudaError_t ce;
  unsigned int* err = device_error_word(c, &ce);
  if (!err) return fail(FA_ERR_CUDA, "device error word: %s", cudaGetErrorString(ce));
  for (int i = 0; i < n; ++i) {
    if ((st = check_layer(c, layers[i]))) return st;
    for (int j = 0; j < i; ++j)
      if (layers[j] == layers[i]) return fail(FA_ERR_INVALID_ARG, "layer %d listed twice", layers[i]);
    const Layer& L = c->layers[layers[i]];
    if (L.owner != layers[i] || T == 0) continue;   // a shared layer stores nothing
    const Slab* s = nullptr;
    if ((st = check_bound(c, layers[i], &s))) return st;
    if (!k[i] || !v[i] || !slot_mapping[i]) return fail(FA_ERR_INVALID_ARG, "k, v, slot_mapping of layer %d must be non-NULL", layers[i]);
    if (!aligned16(k[i]) || !aligned16(v[i])) return fail(FA_ERR_INVALID_ARG, "k, v of layer %d must be 16-byte aligned", layers[i]);
    a[m++] = StoreArgs{k[i], v[i], slot_mapping[i], s->k, s->v, s->k_scale, s->v_scale, T, L.d.num_kv_heads,
                       L.d.head_dim, c->page_size, layer_pages(c, layers[i]), c->kv_dtype,
                       (c->flags & FA_FLAG_EARLY_METADATA) ? 1 : 0, err};
  }
  if (m == 0) return ok();
  ce = launch_store_layers(a, m, static_cast<cudaStream_t>(stream));
  if (ce != cudaSuccess) return fail(FA_ERR_CUDA, "store launch: %s", cudaGetErrorString(ce));
  return ok();
}

namespace fa {
// Plans of the layers of one multi-layer decode launch.  The launch's CTAs
// (two per SM, one wave) are shared among the layers in proportion to their
// tile bounds: with the other layers' CTAs beside them, each layer gets
// fewer and longer CTAs (fewer split merges) than it would launched alone.
static void plan_decode_layers(const fa_cache* c, int n, const int32_t* layers, int B, int max_seq_len,
                               DecodePlan* p) {
  long long tb[FA_MAX_LAYERS_PER_LAUNCH], tot = 0;
  for (int i = 0; i < n; ++i) {
    p[i] = plan_decode(c, layers[i], B, max_seq_len);
    tb[i] = static_cast<long long>(p[i].units) * p[i].max_tiles;
    tot += tb[i];
  }
  const long long slots = 2LL * sm_count();
  for (int i = 0; i < n; ++i) {
    long long share = tot > 0 ? slots * tb[i] / tot : 1;
    if (share < 1) share = 1;
    if (share < p[i].ncta) p[i] = plan_decode(c, layers[i], B, max_seq_len, share);
  }
}
}  // namespace fa

size_t fa_decode_layers_workspace_bytes(const fa_cache* c, int32_t n, const int32_t* layers, int32_t B,
                                        int32_t max_seq_len) {
  if (!c || !layers || n < 1 || n > FA_MAX_LAYERS_PER_LAUNCH || B <= 0 || max_seq_len <= 0) return 0;
  for (int i = 0; i < n; ++i)
    if (check_layer(c, layers[i]) != FA_OK) return 0;
  DecodePlan p[FA_MAX_LAYERS_PER_LAUNCH];
  plan_decode_layers(c, n, layers, B, max_seq_len, p);
  size_t total = 0;
  for (int i = 0; i < n; ++i) total += (p[i].ws_bytes + 255) / 256 * 256;
  return total;
}

namespace fa {
// The launch arguments of one layer's decode (validated by the caller).
static void fill_decode_args(DecodeArgs& a, const fa_cache* c, int32_t layer, const Slab* s, const DecodePlan& p,
                             const void* q, const void* k_new, const void* v_new, const int32_t* slots,
                             const int32_t* block_table, int32_t max_pages_per_seq, const int32_t* seq_lens,
                             int32_t B, int32_t max_seq_len, void* out, float* lse, void* workspace,
                             unsigned int* err) {
  const Layer& L = c->layers[layer];
  a.q = q;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.k = s->k;
  a.v = s->v;
  a.k_new = k_new;
  a.v_new = v_new;
  a.slots = slots;
  a.k_scale = s->k_scale;
  a.v_scale = s->v_scale;
  a.out = out;
  a.lse = lse;
  a.workspace = p.ws_bytes ? workspace : nullptr;
  a.tm_k = &s->tm_kt;
  a.tm_v = &s->tm_vt;
  a.tm_ks = &s->tm_ks;
  a.tm_vs = &s->tm_vs;
  a.B = B;
  a.Hq = L.d.num_q_heads;
  a.Hkv = L.d.num_kv_heads;
  a.D = L.d.head_dim;
  a.kind = L.d.kind;
  a.window = L.d.window;
  a.page_size = c->page_size;
  a.num_pages = layer_pages(c, layer);
  a.max_pages_per_seq = max_pages_per_seq;
  a.max_seq_len = max_seq_len;
  a.kv_dtype = c->kv_dtype;
  a.early_metadata = (c->flags & FA_FLAG_EARLY_METADATA) ? 1 : 0;
  a.sm_scale = L.d.sm_scale;
  a.plan = p;
  a.err = err;
}

// Decode with an optional store of the current token (k_new, v_new, slots
// non-null for an owning layer).
static fa_status decode_call(fa_cache* c, int32_t layer, const void* q, const void* k_new, const void* v_new,
                             const int32_t* slots, const int32_t* block_table, int32_t max_pages_per_seq,
                             const int32_t* seq_lens, int32_t B, int32_t max_seq_len, void* out, float* lse,
                             void* workspace, size_t workspace_bytes, void* stream) {
  fa_status st = check_layer(c, layer);
  if (st) return st;
  if (B < 0) return fail(FA_ERR_INVALID_ARG, "B must be >= 0");
  if (B == 0) return ok();
  const Layer& L = c->layers[layer];
  const Slab* s = nullptr;
  if ((st = check_bound(c, layer, &s))) return st;
  if (!q || !block_table || !seq_lens || !out)
    return fail(FA_ERR_INVALID_ARG, "q, block_table, seq_lens, out must be non-NULL");
  if (!aligned16(q) || !aligned16(out)) return fail(FA_ERR_INVALID_ARG, "q, out must be 16-byte aligned");
  if (max_seq_len < 1) return fail(FA_ERR_INVALID_ARG, "max_seq_len must be >= 1");
  if (max_pages_per_seq < (max_seq_len + c->page_size - 1) / c->page_size)
    return fail(FA_ERR_INVALID_ARG, "max_pages_per_seq %d cannot hold max_seq_len %d", max_pages_per_seq,
                max_seq_len);
  DecodePlan p = plan_decode(c, layer, B, max_seq_len);
  if (workspace_bytes < p.ws_bytes || (p.ws_bytes && !workspace))
    return fail(FA_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", workspace_bytes, p.ws_bytes);
  if (p.ws_bytes && (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(FA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  cudaError_t ce;
  unsigned int* err = device_error_word(c, &ce);
  if (!err) return fail(FA_ERR_CUDA, "device error word: %s", cudaGetErrorString(ce));
  (void)L;
  DecodeArgs a{};
  fill_decode_args(a, c, layer, s, p, q, k_new, v_new, slots, block_table, max_pages_per_seq, seq_lens, B,
                   max_seq_len, out, lse, workspace, err);
  ce = launch_decode(a, static_cast<cudaStream_t>(stream));
  if (ce != cudaSuccess) return fail(FA_ERR_CUDA, "decode launch: %s", cudaGetErrorString(ce));
  return ok();
}

}  // namespace fa

fa_status fa_paged_decode_attn(fa_cache* c, int32_t layer, const void* q, const int32_t* block_table,
                               int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t B,
                               int32_t max_seq_len, void* out, float* lse, void* workspace,
                               size_t workspace_bytes, void* stream) {
  return decode_call(c, layer, q, nullptr, nullptr, nullptr, block_table, max_pages_per_seq, seq_lens, B,
                     max_seq_len, out, lse, workspace, workspace_bytes, stream);
}

fa_status fa_paged_decode_store_attn(fa_cache* c, int32_t layer, const void* q, const void* k_new,
                                     const void* v_new, const int32_t* slot_mapping, const int32_t* block_table,
                                     int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t B,
                                     int32_t max_seq_len, void* out, float* lse, void* workspace,
                                     size_t workspace_bytes, void* stream) {
  fa_status st = check_layer(c, layer);
  if (st) return st;
  if (c->layers[layer].owner != layer)   // a shared layer: its source stored the rows earlier
    return decode_call(c, layer, q, nullptr, nullptr, nullptr, block_table, max_pages_per_seq, seq_lens, B,
                       max_seq_len, out, lse, workspace, workspace_bytes, stream);
  if (B > 0) {
    if (!k_new || !v_new || !slot_mapping)
      return fail(FA_ERR_INVALID_ARG, "k_new, v_new, slot_mapping must be non-NULL for an owning layer");
    if (!aligned16(k_new) || !aligned16(v_new)) return fail(FA_ERR_INVALID_ARG, "k_new, v_new must be 16-byte aligned");
  }
  return decode_call(c, layer, q, k_new, v_new, slot_mapping, block_table, max_pages_per_seq, seq_lens, B,
                     max_seq_len, out, lse, workspace, workspace_bytes, stream);
}

fa_status fa_paged_decode_attn_layers(fa_cache* c, int32_t n, const int32_t* layers, const void* const* q,
                                      const int32_t* const* block_table, int32_t max_pages_per_seq,
                                      const int32_t* seq_lens, int32_t B, int32_t max_seq_len, void* const* out,
                                      float* const* lse, void* workspace, size_t workspace_bytes, void* stream) {
  if (!c) return fail(FA_ERR_INVALID_ARG, "cache is NULL");
  if (n < 1 || n > FA_MAX_LAYERS_PER_LAUNCH) return fail(FA_ERR_INVALID_ARG, "n must be in [1, %d]", FA_MAX_LAYERS_PER_LAUNCH);
  if (!layers || !q || !block_table || !out) return fail(FA_ERR_INVALID_ARG, "layers, q, block_table, out must be non-NULL");
  if (B < 0) return fail(FA_ERR_INVALID_ARG, "B must be >= 0");
  if (!seq_lens) return fail(FA_ERR_INVALID_ARG, "seq_lens must be non-NULL");
  if (max_seq_len < 1) return fail(FA_ERR_INVALID_ARG, "max_seq_len must be >= 1");
  if (max_pages_per_seq < (max_seq_len + c->page_size - 1) / c->page_size)
    return fail(FA_ERR_INVALID_ARG, "max_pages_per_seq %d cannot hold max_seq_len %d", max_pages_per_seq, max_seq_len);
  fa_status st;
  int D = 0;
  for (int i = 0; i < n; ++i) {
    if ((st = check_layer(c, layers[i]))) return st;
    for (int j = 0; j < i; ++j)
      if (layers[j] == layers[i]) return fail(FA_ERR_INVALID_ARG, "layer %d listed twice", layers[i]);
    const int d = c->layers[layers[i]].d.head_dim;
    if (i == 0) D = d;
    else if (d != D) return fail(FA_ERR_UNSUPPORTED, "layers of head_dim %d and %d in one call", D, d);
    if (!q[i] || !block_table[i] || !out[i]) return fail(FA_ERR_INVALID_ARG, "q, block_table, out of layer %d must be non-NULL", layers[i]);
    if (!aligned16(q[i]) || !aligned16(out[i])) return fail(FA_ERR_INVALID_ARG, "q, out of layer %d must be 16-byte aligned", layers[i]);
  }
  if (B == 0) return ok();
  const size_t need = fa_decode_layers_workspace_bytes(c, n, layers, B, max_seq_len);
  if (workspace_bytes < need || (need && !workspace))
    return fail(FA_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", workspace_bytes, need);
  if (need && (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(FA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  cudaError_t ce;
  unsigned int* err = device_error_word(c, &ce);
  if (!err) return fail(FA_ERR_CUDA, "device error word: %s", cudaGetErrorString(ce));
  DecodeArgs a[FA_MAX_LAYERS_PER_LAUNCH];
  DecodePlan plans[FA_MAX_LAYERS_PER_LAUNCH];
  plan_decode_layers(c, n, layers, B, max_seq_len, plans);
  size_t off = 0;
  for (int i = 0; i < n; ++i) {
    const Slab* s = nullptr;
    if ((st = check_bound(c, layers[i], &s))) return st;
    const DecodePlan& p = plans[i];
    a[i] = DecodeArgs{};
    fill_decode_args(a[i], c, layers[i], s, p, q[i], nullptr, nullptr, nullptr, block_table[i], max_pages_per_seq,
                     seq_lens, B, max_seq_len, out[i], lse ? lse[i] : nullptr,
                     p.ws_bytes ? static_cast<char*>(workspace) + off : nullptr, err);
    off += (p.ws_bytes + 255) / 256 * 256;
  }
  ce = launch_decode_layers(a, n, static_cast<cudaStream_t>(stream));
  if (ce != cudaSuccess) return fail(FA_ERR_CUDA, "decode launch: %s", cudaGetErrorString(ce));
  return ok();
}

// The cache's split workspace for an extend launch (mode 0 without one).
static void set_split(const fa_cache* c, ExtendArgs& a) {
  a.split_ws = c->split_ws;
  a.split_cap = c->split_cap;
  a.split_mode = !c->split_ws ? 0 : (c->flags & FA_FLAG_EXTEND_SPLIT_ALL) ? 2 : 1;
}

size_t fa_extend_workspace_bytes(void) { return ext_split_layout(ext_split_cap()).bytes; }

fa_status fa_cache_bind_extend_workspace(fa_cache* c, void* workspace, size_t bytes) {
  if (!c) return fail(FA_ERR_INVALID_ARG, "cache is NULL");
  if (!workspace) {
    c->split_ws = nullptr;
    c->split_cap = 0;
    return ok();
  }
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return fail(FA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  int cap = ext_split_cap();
  while (cap > 0 && ext_split_layout(cap).bytes > bytes) --cap;
  if (cap < 1)
    return fail(FA_ERR_WORKSPACE, "extend workspace %zu bytes < %zu needed for one job", bytes,
                ext_split_layout(1).bytes);
  const cudaError_t ce = cudaMemset(workspace, 0, ext_split_layout(cap).off_ml);   // the arrival counters
  if (ce != cudaSuccess) return fail(FA_ERR_CUDA, "clearing the extend workspace: %s", cudaGetErrorString(ce));
  c->split_ws = workspace;
  c->split_cap = cap;
  return ok();
}

fa_status fa_paged_extend_attn(fa_cache* c, int32_t layer, const void* q, const void* k_ext, const void* v_ext,
                               const int32_t* qo_indptr, const int32_t* prefix_lens, const int32_t* block_table,
                               int32_t max_pages_per_seq, int32_t B, int32_t num_tokens, int32_t max_q_len,
                               int32_t max_prefix_len, void* out, float* lse, void* stream) {
  fa_status st = check_layer(c, layer);
  if (st) return st;
  if (B < 0 || max_q_len < 0 || max_prefix_len < 0 || num_tokens < 0) return fail(FA_ERR_INVALID_ARG, "negative size");
  if (B == 0 || max_q_len == 0 || num_tokens == 0) return ok();
  const Layer& L = c->layers[layer];
  const int g = L.d.num_q_heads / L.d.num_kv_heads;
  if (128 % g != 0)
    return fail(FA_ERR_UNSUPPORTED, "extend packs Hq/Hkv = %d query heads into 128-row tiles; it must divide 128", g);
  const Slab* s = nullptr;
  if ((st = check_bound(c, layer, &s))) return st;
  if (!q || !k_ext || !v_ext || !qo_indptr || !prefix_lens || !out || (max_prefix_len > 0 && !block_table))
    return fail(FA_ERR_INVALID_ARG, "a required pointer is NULL");
  if (!aligned16(q) || !aligned16(k_ext) || !aligned16(v_ext) || !aligned16(out))
    return fail(FA_ERR_INVALID_ARG, "q, k_ext, v_ext, out must be 16-byte aligned");
  if (max_prefix_len > 0 && max_pages_per_seq < (max_prefix_len + c->page_size - 1) / c->page_size)
    return fail(FA_ERR_INVALID_ARG, "max_pages_per_seq %d cannot hold max_prefix_len %d", max_pages_per_seq,
                max_prefix_len);
  cudaError_t ce;
  unsigned int* err = device_error_word(c, &ce);
  if (!err) return fail(FA_ERR_CUDA, "device error word: %s", cudaGetErrorString(ce));
  ExtendArgs a{};
  a.q = q;
  a.k_ext = k_ext;
  a.v_ext = v_ext;
  a.qo_indptr = qo_indptr;
  a.prefix_lens = prefix_lens;
  a.block_table = block_table;
  a.k_slab = s->k;
  a.v_slab = s->v;
  a.k_scale = s->k_scale;
  a.v_scale = s->v_scale;
  a.tm_k = &s->tm_k;
  a.tm_v = &s->tm_v;
  a.tm_ks = &s->tm_ks;
  a.tm_vs = &s->tm_vs;
  a.out = out;
  a.lse = lse;
  a.B = B;
  a.Hq = L.d.num_q_heads;
  a.Hkv = L.d.num_kv_heads;
  a.D = L.d.head_dim;
  a.kind = L.d.kind;
  a.window = L.d.window;
  a.page_size = c->page_size;
  a.num_pages = layer_pages(c, layer);
  a.max_pages_per_seq = max_pages_per_seq;
  a.max_q_len = max_q_len;
  a.max_prefix_len = max_prefix_len;
  a.kv_dtype = c->kv_dtype;
  a.num_tokens = num_tokens;
  a.early_metadata = (c->flags & FA_FLAG_EARLY_METADATA) ? 1 : 0;
  a.sm_scale = L.d.sm_scale;
  a.err = err;
  set_split(c, a);
  if ((st = encode_q_map(&a.tm_q, q, num_tokens, L.d.num_q_heads, L.d.head_dim, g))) return st;
  if ((st = encode_ext_map(&a.tm_kx, k_ext, num_tokens, L.d.num_kv_heads, L.d.head_dim))) return st;
  if ((st = encode_ext_map(&a.tm_vx, v_ext, num_tokens, L.d.num_kv_heads, L.d.head_dim))) return st;
  ce = launch_extend(a, static_cast<cudaStream_t>(stream));
  if (ce != cudaSuccess) return fail(FA_ERR_CUDA, "extend launch: %s", cudaGetErrorString(ce));
  return ok();
}

fa_status fa_paged_decode_multi_attn(fa_cache* c, int32_t layer, const void* q, const int32_t* qo_indptr,
                                     const int32_t* seq_lens, const int32_t* block_table, int32_t max_pages_per_seq,
                                     int32_t B, int32_t num_tokens, int32_t max_q_len, int32_t max_seq_len, void* out,
                                     float* lse, void* stream) {
  fa_status st = check_layer(c, layer);
  if (st) return st;
  if (B < 0 || max_q_len < 0 || max_seq_len < 0 || num_tokens < 0) return fail(FA_ERR_INVALID_ARG, "negative size");
  if (B == 0 || max_q_len == 0 || num_tokens == 0) return ok();
  const Layer& L = c->layers[layer];
  const int g = L.d.num_q_heads / L.d.num_kv_heads;
  if (128 % g != 0)
    return fail(FA_ERR_UNSUPPORTED, "multi-token decode packs Hq/Hkv = %d query heads into 128-row tiles; it must divide 128", g);
  const Slab* s = nullptr;
  if ((st = check_bound(c, layer, &s))) return st;
  if (!q || !qo_indptr || !seq_lens || !block_table || !out) return fail(FA_ERR_INVALID_ARG, "a required pointer is NULL");
  if (!aligned16(q) || !aligned16(out)) return fail(FA_ERR_INVALID_ARG, "q, out must be 16-byte aligned");
  if (max_seq_len < 1) return fail(FA_ERR_INVALID_ARG, "max_seq_len must be >= 1");
  if (max_pages_per_seq < (max_seq_len + c->page_size - 1) / c->page_size)
    return fail(FA_ERR_INVALID_ARG, "max_pages_per_seq %d cannot hold max_seq_len %d", max_pages_per_seq, max_seq_len);
  cudaError_t ce;
  unsigned int* err = device_error_word(c, &ce);
  if (!err) return fail(FA_ERR_CUDA, "device error word: %s", cudaGetErrorString(ce));
  ExtendArgs a{};
  a.q = q;
  a.qo_indptr = qo_indptr;
  a.seq_lens = seq_lens;
  a.keys_in_pages = 1;
  a.block_table = block_table;
  a.k_slab = s->k;
  a.v_slab = s->v;
  a.k_scale = s->k_scale;
  a.v_scale = s->v_scale;
  a.tm_k = &s->tm_k;
  a.tm_v = &s->tm_v;
  a.tm_ks = &s->tm_ks;
  a.tm_vs = &s->tm_vs;
  a.out = out;
  a.lse = lse;
  a.B = B;
  a.Hq = L.d.num_q_heads;
  a.Hkv = L.d.num_kv_heads;
  a.D = L.d.head_dim;
  a.kind = L.d.kind;
  a.window = L.d.window;
  a.page_size = c->page_size;
  a.num_pages = layer_pages(c, layer);
  a.max_pages_per_seq = max_pages_per_seq;
  a.max_q_len = max_q_len;
  a.max_prefix_len = max_seq_len;   // bounds the sequence lengths in this mode
  a.kv_dtype = c->kv_dtype;
  a.num_tokens = num_tokens;
  a.early_metadata = (c->flags & FA_FLAG_EARLY_METADATA) ? 1 : 0;
  a.sm_scale = L.d.sm_scale;
  a.err = err;
  set_split(c, a);
  if ((st = encode_q_map(&a.tm_q, q, num_tokens, L.d.num_q_heads, L.d.head_dim, g))) return st;
  a.tm_kx = s->tm_k;   // no chunk rows in this mode: the chunk maps are never used
  a.tm_vx = s->tm_v;
  ce = launch_extend(a, static_cast<cudaStream_t>(stream));
  if (ce != cudaSuccess) return fail(FA_ERR_CUDA, "decode launch: %s", cudaGetErrorString(ce));
  return ok();
}

}  // extern "C"
