// Internal declarations shared by the host API and the kernel launchers.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <vector>

#include "fa.h"

namespace fa {

// Token rows are processed in 16-row tiles: one m16 tile of the warp MMAs and
// one TMA box height.  Page sizes are multiples of it.
constexpr int kTile = 16;
// Layers one multi-layer launch can hold.
constexpr int kMaxLayersPerLaunch = FA_MAX_LAYERS_PER_LAUNCH;

struct Slab {
  void* k = nullptr;
  void* v = nullptr;
  float* k_scale = nullptr;
  float* v_scale = nullptr;
  bool bound = false;
  // TMA descriptors over K and V, 3-D: (64-element column block, block index,
  // row) with rows = num_pages * Hkv * page_size; see fa_cache_bind_slab.
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  // The same slabs as (column-block element, row, column block): one box is
  // a whole 16-row tile, all column blocks, landing block-major like 16-row
  // boxes of tm_k / tm_v side by side (one copy per tile).
  CUtensorMap tm_kt;
  CUtensorMap tm_vt;
  // int8 format: 2-D maps over the fp32 scales, one 16-float box per tile.
  CUtensorMap tm_ks;
  CUtensorMap tm_vs;
};

struct Layer {
  fa_layer_desc d;
  int owner = -1;   // slab owner (itself if it owns a slab)
};

}  // namespace fa

struct fa_cache {
  std::vector<fa::Layer> layers;
  std::vector<fa::Slab> slabs;   // indexed by layer; only owners are bound
  int32_t num_pages = 0;      // pages of each full layer's slab
  int32_t window_pages = 0;   // pages of each sliding layer's slab (0: num_pages)
  int32_t page_size = 0;
  int32_t kv_dtype = FA_KV_BF16;
  uint32_t flags = 0;   // FA_FLAG_*
  int32_t err_slot = -1;   // this cache's device error word (index into the per-device array)
  void* split_ws = nullptr;   // extend split workspace (caller's memory), split_cap jobs
  int32_t split_cap = 0;
};

namespace fa {

// Pages in the slab a layer reads: sliding layers may have a pool of their own.
inline int32_t layer_pages(const fa_cache* c, int32_t layer) {
  return (c->layers[layer].d.kind == FA_SLIDING && c->window_pages > 0) ? c->window_pages : c->num_pages;
}

// thread-local error message
fa_status fail(fa_status st, const char* fmt, ...);

// The cache's device error word on the current device (file-scope
// __device__ storage, one word per live cache), and its synchronous clear.
unsigned int* device_error_word(const fa_cache* c, cudaError_t* err);
cudaError_t clear_device_error_word(const fa_cache* c);

int sm_count();

// Set a kernel's dynamic shared-memory limit once per device.
cudaError_t set_smem_once(const void* fn, int bytes, unsigned int* done_mask);

// ---------------------------------------------------------------- decode plan
// The decode kernel splits the concatenated tile lists of all (sequence, KV
// head, head chunk) units evenly over at most `ncta` CTAs; a unit whose tiles
// land on one CTA is finished there, the others are merged by the last CTA of
// the unit to finish (an arrival counter per unit lives in the workspace).
struct DecodePlan {
  int head_chunks = 1;      // ceil(g / 8): query heads are packed 8 per MMA column block
  int units = 0;            // B * Hkv * head_chunks
  int max_tiles = 0;        // 16-row tiles a unit can touch under the length bound
  int min_tiles = 0;        // fewest tiles a CTA is given
  int ncta = 0;             // CTAs launched
  size_t off_ml = 0, off_o = 0;   // workspace layout (bytes); counters [units] at 0
  size_t ws_bytes = 0;
};
// max_cta > 0 caps the launch's CTAs for this layer (default: two per SM).
DecodePlan plan_decode(const fa_cache* c, int layer, int B, int max_seq_len, long long max_cta = 0);

// Launch with programmatic stream serialisation (overlaps launch latency with
// the previous kernel's tail); every kernel waits on griddepcontrol first.
bool pdl_enabled();

template <typename Kern, typename... Args>
static cudaError_t launch_pdl(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

struct StoreArgs {
  const void* k;
  const void* v;
  const int32_t* slots;
  void* k_slab;
  void* v_slab;
  float* k_scale;
  float* v_scale;
  int T, Hkv, D, page_size, num_pages, kv_dtype, early_metadata;
  unsigned int* err;
};
cudaError_t launch_store(const StoreArgs& a, cudaStream_t s);
// The stores of several layers in one launch (n <= kMaxLayersPerLaunch; any head_dim mix).
cudaError_t launch_store_layers(const StoreArgs* a, int n, cudaStream_t s);

struct DecodeArgs {
  const void* q;
  const int32_t* block_table;
  const int32_t* seq_lens;
  const void* k;   // slab bases (L2 prefetch, the current token's store)
  const void* v;
  const void* k_new;        // fused store of the current token (null: none)
  const void* v_new;
  const int32_t* slots;
  const float* k_scale;
  const float* v_scale;
  void* out;
  float* lse;
  void* workspace;
  const CUtensorMap* tm_k;
  const CUtensorMap* tm_v;
  const CUtensorMap* tm_ks;
  const CUtensorMap* tm_vs;
  int B, Hq, Hkv, D, kind, window, page_size, num_pages, max_pages_per_seq, max_seq_len, kv_dtype;
  int early_metadata;
  float sm_scale;
  DecodePlan plan;
  unsigned int* err;
};
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s);
// Several layers of one head_dim and KV format in one launch (n <= kMaxLayersPerLaunch).
cudaError_t launch_decode_layers(const DecodeArgs* a, int n, cudaStream_t s);

struct ExtendArgs {
  const void* q;
  const void* k_ext;
  const void* v_ext;
  const int32_t* qo_indptr;
  const int32_t* prefix_lens;
  const int32_t* seq_lens;   // keys_in_pages: lengths including the new tokens
  const int32_t* block_table;
  const void* k_slab;
  const void* v_slab;
  const float* k_scale;
  const float* v_scale;
  const CUtensorMap* tm_k;
  const CUtensorMap* tm_v;
  const CUtensorMap* tm_ks;
  const CUtensorMap* tm_vs;
  void* out;
  float* lse;
  int B, Hq, Hkv, D, kind, window, page_size, num_pages, max_pages_per_seq, max_q_len,
      max_prefix_len, kv_dtype, num_tokens, early_metadata;
  int keys_in_pages;   // 1: every key from the slab (new tokens already stored), no k_ext / v_ext
  float sm_scale;
  unsigned int* err;
  // per-call maps: q as (64-column block, head, token, block index) boxes of
  // (64, g, 128/g, 1); k_ext / v_ext as (64, block, KV head, token) boxes of (64, 1, 1, 64)
  CUtensorMap tm_q, tm_kx, tm_vx;
  // the cache's split workspace (null: none), the jobs it holds, and the
  // mode: 0 no split, 1 the last wave's jobs when that wave is at most half
  // full and the jobs are long, 2 the last split_cap jobs whatever their size
  void* split_ws;
  int split_cap, split_mode;
};
cudaError_t launch_extend(const ExtendArgs& a, cudaStream_t s);

// Split workspace of extend for `cap` jobs: arrival counters, then per job
// and CTA 128 rows of (base, rounded sum, unrounded sum, 0), then per job
// and CTA a 128 x 256 fp32 partial O; each part 256-byte aligned.
struct ExtSplitLayout {
  size_t off_ml, off_o, bytes;
};
inline ExtSplitLayout ext_split_layout(int cap) {
  auto up = [](size_t b) { return (b + 255) / 256 * 256; };
  ExtSplitLayout l;
  l.off_ml = up(static_cast<size_t>(cap) * sizeof(int));
  l.off_o = l.off_ml + up(static_cast<size_t>(cap) * 2 * 128 * 16);
  l.bytes = l.off_o + static_cast<size_t>(cap) * 2 * 128 * 256 * sizeof(float);
  return l;
}
// Jobs the split workspace of this device holds: half the SMs (the largest
// last wave worth splitting in two).
inline int ext_split_cap() {
  const int n = sm_count() / 2;
  return n > 0 ? n : 1;
}

}  // namespace fa
