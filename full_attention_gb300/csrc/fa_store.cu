// Paged KV store: scatter post-RoPE k, v rows of new tokens into their slots
// ("FreeToken PR #898", description bullet on store_kv; "unsloth commit
// dee9371": the store layer writes its post-rotary k, v into its paged cache).
//
// One warp moves one (token, KV head, K-or-V) row with 16-byte vector loads
// and stores.  The 8-bit per-token-head formats quantise the row on the way:
// a = max|x| (fp32, warp-shuffle reduction); int8: s = a / 127, c = rint(x / s)
// clamped to [-127, 127]; fp8: s = a / 448, c = the e4m3 value nearest x / s,
// saturating at 448; every division IEEE round-to-nearest.
#include <algorithm>
#include <cstdio>
#include <mutex>

#include "fa_internal.h"
#include "fa_ptx.cuh"
#include "fa_row.cuh"

// Device error words: one per live cache descriptor (the cache's slot), where
// every kernel a call on that cache launches ORs its FA_DEV_ERR_* bits.
// File-scope device storage: nothing is allocated for them.
__device__ unsigned int g_fa_device_error[FA_MAX_CACHES];

namespace fa {

// Base of the error words on the current device.  In host code the array's
// name is a host-side stand-in, so its device address is looked up once per
// device, with that device current.
static unsigned int* device_error_words(cudaError_t* err) {
  static std::mutex mu;
  static unsigned int* ptrs[128] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 128) {
    *err = e != cudaSuccess ? e : cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_fa_device_error);
    if (e != cudaSuccess) {
      *err = e;
      return nullptr;
    }
    ptrs[dev] = static_cast<unsigned int*>(p);
  }
  *err = cudaSuccess;
  return ptrs[dev];
}

unsigned int* device_error_word(const fa_cache* c, cudaError_t* err) {
  unsigned int* base = device_error_words(err);
  return base ? base + c->err_slot : nullptr;
}

cudaError_t clear_device_error_word(const fa_cache* c) {
  cudaError_t e;
  unsigned int* w = device_error_word(c, &e);
  if (!w) return e;
  const unsigned int zero = 0;
  return cudaMemcpy(w, &zero, sizeof(zero), cudaMemcpyHostToDevice);
}

// R consecutive (token, KV head, K or V) rows per warp, `warp` counting the
// launch's warps for this layer.  The warp loads the R slots, then (once the
// previous kernel's rows may be read) all R rows, whose addresses do not
// depend on the slots, then stores them: R * D / 256 16-byte vectors per lane
// in flight behind one load latency.  Row t * Hkv * 2 + 2 h (+1) is token t's
// K (V) row of KV head h.
template <int D>
struct StoreShape {
  static constexpr int R = D == 256 ? 8 : 4;   // rows per warp: 128 bytes per lane in flight
};

template <int D, int KV>
__device__ __forceinline__ void store_rows(const StoreArgs& a, int warp, int lane) {
  constexpr int R = StoreShape<D>::R;
  const int rows = a.T * a.Hkv * 2;
  const int r0 = warp * R;
  if (r0 >= rows) return;
  int slot[R];
#pragma unroll
  for (int i = 0; i < R; ++i) slot[i] = (r0 + i < rows) ? __ldg(a.slots + ((r0 + i) >> 1) / a.Hkv) : -1;
  griddep_wait();   // the rows (and the slab) may belong to the previous kernel
  RowRegs<D> r[R];
#pragma unroll
  for (int i = 0; i < R; ++i)
    if (r0 + i < rows)
      row_load<D>(r[i], static_cast<const __nv_bfloat16*>(((r0 + i) & 1) ? a.v : a.k) +
                            static_cast<size_t>((r0 + i) >> 1) * D, lane);
  constexpr size_t elem = KV == FA_KV_BF16 ? 2 : 1;
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const int row = r0 + i;
    if (row >= rows || slot[i] < 0) continue;   // a negative slot is a padding token
    const int page = slot[i] / a.page_size, off = slot[i] % a.page_size;
    if (page >= a.num_pages) {
      if (lane == 0) atomicOr(a.err, FA_DEV_ERR_SLOT);
      continue;
    }
    const int h = (row >> 1) % a.Hkv;
    const size_t dst = (static_cast<size_t>(page) * a.Hkv + h) * a.page_size + off;
    const int which = row & 1;
    row_store<D, KV>(r[i], static_cast<uint8_t*>(which ? a.v_slab : a.k_slab) + dst * D * elem,
                     KV == FA_KV_BF16 ? nullptr : (which ? a.v_scale : a.k_scale) + dst, lane);
  }
}

template <int D, int KV>
__global__ void __launch_bounds__(256) store_kernel(StoreArgs a) {
  if (!a.early_metadata) griddep_wait();
  griddep_launch_dependents();
  store_rows<D, KV>(a, (blockIdx.x * blockDim.x + threadIdx.x) >> 5, threadIdx.x & 31);
}

// Several layers' stores in one launch: blockIdx.y picks the layer.
struct StoreLayers {
  StoreArgs a[kMaxLayersPerLaunch];
};

template <int KV>
__global__ void __launch_bounds__(256) store_layers_kernel(const __grid_constant__ StoreLayers m) {
  const StoreArgs& a = m.a[blockIdx.y];
  if (!a.early_metadata) griddep_wait();
  griddep_launch_dependents();
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (a.D == 256) store_rows<256, KV>(a, warp, lane);
  else store_rows<512, KV>(a, warp, lane);
}

// Warps a store of T tokens needs.
static long store_warps(const StoreArgs& a) {
  const long rows = static_cast<long>(a.T) * a.Hkv * 2;
  const int R = a.D == 256 ? StoreShape<256>::R : StoreShape<512>::R;
  return (rows + R - 1) / R;
}

cudaError_t launch_store_layers(const StoreArgs* a, int n, cudaStream_t s) {
  if (n < 1 || n > kMaxLayersPerLaunch) return cudaErrorInvalidValue;
  StoreLayers m{};
  long warps = 0;
  for (int i = 0; i < n; ++i) {
    m.a[i] = a[i];
    warps = std::max(warps, store_warps(a[i]));
  }
  const int block = 256;
  const long grid = (warps * 32 + block - 1) / block;
  if (grid > 0x7fffffffL) return cudaErrorInvalidValue;
  const dim3 g(static_cast<unsigned>(grid), static_cast<unsigned>(n)), b(block);
  if (a[0].kv_dtype == FA_KV_INT8) return launch_pdl(store_layers_kernel<FA_KV_INT8>, g, b, 0, s, m);
  if (a[0].kv_dtype == FA_KV_FP8) return launch_pdl(store_layers_kernel<FA_KV_FP8>, g, b, 0, s, m);
  return launch_pdl(store_layers_kernel<FA_KV_BF16>, g, b, 0, s, m);
}

cudaError_t launch_store(const StoreArgs& a, cudaStream_t s) {
  const long warps = store_warps(a);
  const int block = 256;
  const long grid = (warps * 32 + block - 1) / block;
  if (grid > 0x7fffffffL) return cudaErrorInvalidValue;
  const dim3 g(static_cast<unsigned>(grid)), b(block);
  if (a.kv_dtype == FA_KV_INT8)
    return a.D == 256 ? launch_pdl(store_kernel<256, FA_KV_INT8>, g, b, 0, s, a)
                      : launch_pdl(store_kernel<512, FA_KV_INT8>, g, b, 0, s, a);
  if (a.kv_dtype == FA_KV_FP8)
    return a.D == 256 ? launch_pdl(store_kernel<256, FA_KV_FP8>, g, b, 0, s, a)
                      : launch_pdl(store_kernel<512, FA_KV_FP8>, g, b, 0, s, a);
  return a.D == 256 ? launch_pdl(store_kernel<256, FA_KV_BF16>, g, b, 0, s, a)
                    : launch_pdl(store_kernel<512, FA_KV_BF16>, g, b, 0, s, a);
}

}  // namespace fa

extern "C" fa_status fa_get_device_error(fa_cache* cache, int32_t* code, void* stream) {
  if (!cache) return fa::fail(FA_ERR_INVALID_ARG, "cache is NULL");
  if (!code) return fa::fail(FA_ERR_INVALID_ARG, "code is NULL");
  cudaError_t ce;
  unsigned int* p = fa::device_error_word(cache, &ce);
  if (!p) return fa::fail(FA_ERR_CUDA, "device error word: %s", cudaGetErrorString(ce));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned int v = 0;
  if ((ce = cudaStreamSynchronize(s)) != cudaSuccess ||
      (ce = cudaMemcpyAsync(&v, p, sizeof(v), cudaMemcpyDeviceToHost, s)) != cudaSuccess ||
      (ce = cudaMemsetAsync(p, 0, sizeof(v), s)) != cudaSuccess || (ce = cudaStreamSynchronize(s)) != cudaSuccess)
    return fa::fail(FA_ERR_CUDA, "reading the device error word: %s", cudaGetErrorString(ce));
  *code = static_cast<int32_t>(v);
  return FA_OK;
}
