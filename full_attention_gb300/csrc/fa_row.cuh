// One (token, KV head) row of k or v moved into its slab row by one warp:
// bf16 copied verbatim, or quantised to an 8-bit per-token-head format
// ("FreeToken PR #898", description: one fp32 scale per token and head;
// int8 codes in [-127, 127], or fp8 e4m3 codes).  Used by the store kernel and by the decode kernel
// that stores the current token itself, so both write identical bytes.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cstdint>

#include "fa.h"

namespace fa {

template <int D>
struct RowRegs {
  static constexpr int NV = D / 256;   // 16-byte vectors (8 bf16) per lane
  uint4 v[NV];
};

template <int D>
__device__ __forceinline__ void row_load(RowRegs<D>& r, const __nv_bfloat16* src, int lane) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int i = 0; i < RowRegs<D>::NV; ++i) r.v[i] = __ldg(s + i * 32 + lane);
}

template <int D>
__device__ __forceinline__ void row_store_bf16(const RowRegs<D>& r, __nv_bfloat16* dst, int lane) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < RowRegs<D>::NV; ++i) d[i * 32 + lane] = r.v[i];
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float (&x)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// a = max |x| (fp32), s = a / 127, c = rint(x / s) clamped to [-127, 127],
// both divisions IEEE round-to-nearest; a = 0 gives s = 0 and all-zero codes.
// Lane l holds values [i * 256 + 8 l, i * 256 + 8 l + 8) of the row.
template <int D>
__device__ __forceinline__ void row_store_int8(const RowRegs<D>& r, int8_t* dst, float* scale, int lane) {
  constexpr int NV = RowRegs<D>::NV;
  float x[NV][8];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    bf16x8_to_f32(r.v[i], x[i]);
#pragma unroll
    for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(x[i][e]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float s = __fdiv_rn(amax, 127.0f);
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    uint32_t packed[2] = {0u, 0u};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      int c = 0;
      if (amax != 0.0f) {
        float qv = rintf(__fdiv_rn(x[i][e], s));
        qv = fminf(fmaxf(qv, -127.0f), 127.0f);
        c = static_cast<int>(qv);
      }
      packed[e >> 2] |= (static_cast<uint32_t>(c) & 0xffu) << (8 * (e & 3));
    }
    *reinterpret_cast<uint2*>(dst + i * 256 + lane * 8) = make_uint2(packed[0], packed[1]);
  }
  if (lane == 0) *scale = s;
}

// a = max |x| (fp32), s = a / 448 (IEEE), c = the e4m3 value nearest to the
// IEEE quotient x / s, ties to the even mantissa, saturating at the largest
// finite magnitude 448; a = 0 gives s = 0 and all-zero codes.  Same lane
// layout as row_store_int8.
template <int D>
__device__ __forceinline__ void row_store_fp8(const RowRegs<D>& r, uint8_t* dst, float* scale, int lane) {
  constexpr int NV = RowRegs<D>::NV;
  float x[NV][8];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    bf16x8_to_f32(r.v[i], x[i]);
#pragma unroll
    for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(x[i][e]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float s = __fdiv_rn(amax, 448.0f);
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    uint32_t packed[2] = {0u, 0u};
    if (amax != 0.0f) {
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        const float2 qv = make_float2(__fdiv_rn(x[i][e], s), __fdiv_rn(x[i][e + 1], s));
        // element e in the lower byte of the pair
        const uint32_t pair = __nv_cvt_float2_to_fp8x2(qv, __NV_SATFINITE, __NV_E4M3);
        packed[e >> 2] |= (pair & 0xffffu) << (8 * (e & 3));
      }
    }
    *reinterpret_cast<uint2*>(dst + i * 256 + lane * 8) = make_uint2(packed[0], packed[1]);
  }
  if (lane == 0) *scale = s;
}

// The slab format's per-row store: KV is the fa_kv_dtype of the slab.
template <int D, int KV>
__device__ __forceinline__ void row_store(const RowRegs<D>& r, void* dst, float* scale, int lane) {
  if constexpr (KV == FA_KV_BF16) row_store_bf16<D>(r, static_cast<__nv_bfloat16*>(dst), lane);
  else if constexpr (KV == FA_KV_INT8) row_store_int8<D>(r, static_cast<int8_t*>(dst), scale, lane);
  else row_store_fp8<D>(r, static_cast<uint8_t*>(dst), scale, lane);
}

}  // namespace fa
