// Paged decode attention: balanced split-K online softmax, GQA-packed.
//
// Regimes ("unsloth gemma4_flex_inference.py" history, commit "block mask per
// attention regime"; "pegainfer issue #807", Description): a full layer's
// query at q_pos = L - 1 sees keys [0, q_pos]; a sliding layer's sees
// [max(0, L - W), q_pos].  Sliding layers only visit the 16-row tiles that
// hold in-window keys.  KV-shared layers arrive here with their source's slab
// ("FreeToken PR #898", description).
//
// Work decomposition.  A unit is (sequence, KV head, chunk of up to 8 query
// heads); its work is the list of 16-row tiles its query can see.  The tile
// lists of all units are laid end to end and cut into equal contiguous
// shares, one per CTA (at most two CTAs per SM, one wave), so every CTA moves
// the same number of bytes whatever the length mix.  A CTA walks its share
// unit segment by unit segment without draining its pipeline.  A unit whose
// tiles all fall on one CTA is finished there; the others leave per-CTA
// partial (max, sum, o) rows, and the last of their CTAs to arrive (counted
// by an atomic per unit in the workspace) merges them.
//
// Per tile the contraction is
//   S^T (16 keys x 8 heads)  = K (16 x D) . Q^T (D x 8)         (mma.sync m16n8k16)
//   O^T (D x 8 heads)       += V^T (D x 16) . P^T (16 x 8)
// with keys on the MMA M side, so 8 query heads fill N exactly and each KV
// byte is read from HBM once for the whole group.  Warp 4 is a TMA producer:
// it streams K and V tiles (and 8-bit scales) into a 3-stage ring of
// 128-byte-swizzled shared-memory tiles, and each segment's queries by a bulk
// copy.  Warps 0-3 split the QK^T contraction over columns, exchange partial
// scores through shared memory, run the online softmax redundantly (each lane
// owns one head) and each accumulate a quarter of O's columns.
//
// bf16 slabs use bf16 MMAs.  int8 and fp8 slabs: codes become exact fp16
// values (int8: byte permute + one subtraction; e4m3: the hardware pair
// conversion), the K scale multiplies the fp32 scores, the V scale is folded
// into P (normalised by the step's largest scale, which joins the running
// rescale), and the MMAs run in fp16; a query element f16 cannot hold
// (magnitude 65536 or more) saturates to +-65504 and sets FA_DEV_ERR_RANGE.
#include <cfloat>
#include <climits>
#include <mutex>

#include "fa_internal.h"
#include "fa_ptx.cuh"
#include "fa_row.cuh"

namespace fa {

template <int D, int KV>
struct DecCfg {
  static constexpr int ELEM = KV ? 1 : 2;
  static constexpr int ROWB = D * ELEM;                 // bytes per row
  static constexpr int NBLK = ROWB / 128;               // 128-byte column blocks per row
  static constexpr int TILE_BYTES = kTile * ROWB;       // one 16-row tile of K (or V)
  // tiles per pipeline step: 32 KB of K+V, but at most 2, since more tiles
  // per step lengthen the consumer chain between barriers (8-bit head_dim
  // 256 measured 2% faster at 2 tiles than at 4, slower at 1)
  static constexpr int NT = 32768 / (2 * TILE_BYTES) < 2 ? 32768 / (2 * TILE_BYTES) : 2;
  static constexpr int NSTAGE = 3;
  static constexpr int PREFETCH_TILES = 2 * NSTAGE * NT; // tiles a CTA pulls into L2 before its dependency resolves
  static constexpr int NCW = 4;                         // consumer warps
  static constexpr int NTHR = (NCW + 1) * 32;
  static constexpr int QK_COLS = D * NT / NCW;          // QK^T columns per warp
  static constexpr int PV_COLS = D / NCW;               // output columns per warp
  static constexpr int PV_MT = PV_COLS / 16;            // m16 tiles of O^T per warp
  static constexpr int STAGE_KV = 2 * NT * TILE_BYTES;
  static constexpr int SC_BYTES = KV ? 2 * NT * 128 : 0; // k, v scales of the step's tiles (128-B slots)
  static constexpr int SX_STRIDE = 12;                  // floats per key row (bank-conflict free)
  static constexpr int SX_BYTES = 2 * NCW * kTile * SX_STRIDE * 4;
  static constexpr int Q_BYTES = 8 * D * 2;             // one segment's queries, bf16 [8][D]
  static constexpr int OFF_SC = NSTAGE * STAGE_KV;
  static constexpr int OFF_Q = OFF_SC + NSTAGE * SC_BYTES;
  static constexpr int OFF_SX = OFF_Q + Q_BYTES;
  static constexpr int OFF_BAR = OFF_SX + SX_BYTES;
  static constexpr int SMEM = OFF_BAR + (2 * NSTAGE + 3) * 8;
  static constexpr int STAGE_ALL = NSTAGE * STAGE_KV;   // the ring, reused to stage a merge
  static constexpr int SMEM_ALLOC = SMEM + 1024;
  static_assert(NT >= 1 && NCW % NT == 0 && 32 % NT == 0, "step shape");
  static_assert(QK_COLS % 32 == 0 && PV_COLS % 32 == 0, "warp column split");
};

struct DecK {
  const __nv_bfloat16* q;
  const int32_t* block_table;
  const int32_t* seq_lens;
  uint8_t* kb;    // slab bases and int8 scales (L2 prefetch, the current token's store)
  uint8_t* vb;
  float* ksb;
  float* vsb;
  const __nv_bfloat16* k_new;   // current token's rows [B][Hkv][D] and their slots, stored by
  const __nv_bfloat16* v_new;   // the CTA that reads the unit's last tile (null: no store)
  const int32_t* slots;
  __nv_bfloat16* out;
  float* lse;
  int* counters;    // [U] arrival count per unit (null: no workspace, one CTA); zero between calls
  float* ml_part;   // [(ncta + U) * 8][2]
  float* o_part;    // [(ncta + U) * 8][D]
  unsigned int* err;
  int B, Hq, Hkv, g, chunks, kind, window, page_size, tiles_per_page, num_pages, max_pages_per_seq;
  int max_seq_len, units, min_tiles, early_metadata;
  float scale_log2;   // sm_scale * log2(e)
};

struct Unit {
  int b, h, c, L, lo, t_first, n;
};

__device__ __forceinline__ Unit unit_of(const DecK& p, int u) {
  Unit x;
  x.b = u / (p.Hkv * p.chunks);
  const int r = u % (p.Hkv * p.chunks);
  x.h = r / p.chunks;
  x.c = r % p.chunks;
  const int L = __ldg(p.seq_lens + x.b);
  x.L = min(L, p.max_seq_len);
  if (x.L <= 0) {
    x.lo = x.t_first = x.n = 0;
    return x;
  }
  x.lo = (p.kind == FA_SLIDING) ? max(0, x.L - p.window) : 0;
  x.t_first = x.lo / kTile;
  x.n = (x.L - 1) / kTile + 1 - x.t_first;
  return x;
}

// CTA that owns global tile g when T tiles are split evenly over n CTAs.
__device__ __forceinline__ int cta_of(long long g, int n, long long T) {
  return static_cast<int>(((g + 1) * n - 1) / T);
}

// int8 x4 (a 32-bit word, bias-xored) -> fp16x2 holding two exact integers.
// sel picks the bytes: 0x4140 -> (b0, b1), 0x4342 -> (b2, b3), 0x4240 -> (b0, b2), 0x4341 -> (b1, b3).
__device__ __forceinline__ uint32_t i8pair_to_f16x2(uint32_t biased, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(biased), "r"(0x64646464u), "r"(sel));
  // (0x64 << 8 | u) as fp16 is 1024 + u with u = c + 128; subtract 1152 to get c.
  __half2 h = *reinterpret_cast<__half2*>(&r);
  h = __hsub2(h, __half2(__float2half(1152.0f), __float2half(1152.0f)));
  return *reinterpret_cast<uint32_t*>(&h);
}

// f16x2 of code bytes I (lower half) and J (upper half) of `raw`: int8 codes
// or fp8 e4m3 codes, both exact in f16 (e4m3's 3-bit mantissa and its range
// 2^-9 .. 448 lie inside f16's normal numbers).
template <int KV, int I, int J>
__device__ __forceinline__ uint32_t codes_to_f16x2(uint32_t raw) {
  if constexpr (KV == FA_KV_INT8) {
    return i8pair_to_f16x2(raw ^ 0x80808080u, I | 0x40u | (J << 8) | 0x4000u);
  } else {
    const uint32_t two = (I == 0 && J == 1) ? (raw & 0xffffu)
                         : (I == 2 && J == 3) ? (raw >> 16) : __byte_perm(raw, 0u, I | (J << 4));
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two), __NV_E4M3);
    return static_cast<uint32_t>(h.x) | (static_cast<uint32_t>(h.y) << 16);
  }
}

// Exclusive block scan over all threads of the block; *total gets the sum.
__device__ __forceinline__ int block_excl_scan(int v, int* sm, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) sm[warp] = incl;
  __syncthreads();
  int base = 0, tot = 0;
  for (int w = 0; w < nw; ++w) {
    if (w < warp) base += sm[w];
    tot += sm[w];
  }
  __syncthreads();
  *total = tot;
  return base + incl - v;
}

// Block-wide (min, max) of one value per thread; sm holds 2 ints per warp.
__device__ __forceinline__ int2 block_min_max(int mn, int mx, int* sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  if (lane == 0) {
    sm[2 * warp] = mn;
    sm[2 * warp + 1] = mx;
  }
  __syncthreads();
  int a = sm[0], b = sm[1];
  for (int w = 1; w < nw; ++w) {
    a = min(a, sm[2 * w]);
    b = max(b, sm[2 * w + 1]);
  }
  __syncthreads();
  return make_int2(a, b);
}

// Sequences of length <= 0 get out = 0 and lse = -inf; CTA `cta` of `ncta`
// writes the units u with u % ncta == cta.
// The current token's K and V rows of (sequence b, KV head h) into slot `slot`
// (one warp; slot < 0 skips, a slot past the pool is reported).
template <int D, int KV>
__device__ __forceinline__ void store_current(const DecK& p, const RowRegs<D>& rk, const RowRegs<D>& rv, int h,
                                              int slot, int lane) {
  if (slot < 0) return;
  const int page = slot / p.page_size, off = slot % p.page_size;
  if (page >= p.num_pages) {
    if (lane == 0) atomicOr(p.err, FA_DEV_ERR_SLOT);
    return;
  }
  const size_t row = (static_cast<size_t>(page) * p.Hkv + h) * p.page_size + off;
  constexpr size_t elem = KV == FA_KV_BF16 ? 2 : 1;
  row_store<D, KV>(rk, p.kb + row * D * elem, KV == FA_KV_BF16 ? nullptr : p.ksb + row, lane);
  row_store<D, KV>(rv, p.vb + row * D * elem, KV == FA_KV_BF16 ? nullptr : p.vsb + row, lane);
}

template <int D, int KV>
__device__ void zero_empty_units(const DecK& p, int cta, int ncta, int tid, int nthr) {
  for (int u = cta; u < p.units; u += ncta) {
    const Unit x = unit_of(p, u);
    if (x.L > 0) continue;
    if (p.slots && x.c == 0 && tid < 32) {   // nothing to attend, but the row is still stored
      RowRegs<D> rk, rv;
      const size_t src = (static_cast<size_t>(x.b) * p.Hkv + x.h) * D;
      row_load<D>(rk, p.k_new + src, tid);
      row_load<D>(rv, p.v_new + src, tid);
      store_current<D, KV>(p, rk, rv, x.h, __ldg(p.slots + x.b), tid);
    }
    const int nh = min(8, p.g - x.c * 8), head0 = x.h * p.g + x.c * 8;
    for (int i = tid; i < nh * D; i += nthr)
      p.out[(static_cast<size_t>(x.b) * p.Hq + head0 + i / D) * D + i % D] = __float2bfloat16(0.0f);
    if (p.lse && tid < nh) p.lse[static_cast<size_t>(x.b) * p.Hq + head0 + tid] = -INFINITY;
  }
}

// Merge the partial rows of unit u that CTAs cf..cl left (this CTA arrived
// last): per head h, M = max_c m_c, L = sum_c l_c 2^(m_c - M) and
// out = sum_c o_c 2^(m_c - M) / L, lse = (M + log2 L) ln 2.  Run by the 128
// consumer threads; wbuf is shared scratch of 8 * 128 + 16 floats.  Loads are
// batched so that a typical merge (a handful of source CTAs) costs a few L2
// round trips.
template <int D, int STAGE_BYTES>
__device__ void merge_unit(const DecK& p, int u, const Unit& x, int nh, int head0, int cf, int cl, float* wbuf,
                           uint8_t* stage, uint64_t* sbar, volatile int* abort_flag) {
  constexpr int CH = 128;                  // source CTAs per weight chunk
  constexpr int ITEMS = 8 * (D / 4) / 128; // float4 outputs per thread
  constexpr int ROW_BYTES = 8 * D * 4;     // one source's o rows
  constexpr int NB = STAGE_BYTES / ROW_BYTES;   // sources per staged batch
  const int tid = threadIdx.x;
  const int nct = cl - cf + 1;
  // Staged path (the ring is idle and every weight fits one chunk): bulk
  // copies bring NB sources' o rows into shared memory per batch, so a merge
  // costs one L2 round trip per batch instead of one per source.
  const bool staged = stage != nullptr && nct <= CH;
  auto stage_batch = [&](int b0, int batch) {   // thread 0: request sources b0 .. b0 + n - 1
    const int n = min(NB, nct - b0);
    mbar_arrive_expect_tx(sbar, n * ROW_BYTES);
    for (int c = 0; c < n; ++c)
      bulk_load(stage + c * ROW_BYTES, p.o_part + (static_cast<size_t>(cf + b0 + c) + u) * 8 * D, ROW_BYTES, sbar);
    (void)batch;
  };
  if (staged && tid == 0) {
    fence_proxy_async_global();   // the other CTAs' rows, seen through the acquire, for the bulk copies
    stage_batch(0, 0);
  }
  const float2* mlg = reinterpret_cast<const float2*>(p.ml_part);
  float* Mh = wbuf + 8 * CH;
  float* Lh = Mh + 8;
  const int h = tid >> 4, k = tid & 15;    // 16 threads per head
  // one pass: running max with rescaled sum; the first 64 pairs stay in
  // registers for the weights
  float M = -INFINITY, L = 0.f;
  float2 v[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int c = k + 16 * r;
    v[r] = c < nct ? __ldcg(mlg + (static_cast<size_t>(cf + c) + u) * 8 + h) : make_float2(-INFINITY, 0.f);
  }
  auto fold = [&](float2 x) {
    if (x.x == -INFINITY) return;
    const float Mn = fmaxf(M, x.x);
    L = L * ex2(M - Mn) + x.y * ex2(x.x - Mn);
    M = Mn;
  };
#pragma unroll
  for (int r = 0; r < 4; ++r) fold(v[r]);
  for (int c = k + 64; c < nct; c += 16) fold(__ldcg(mlg + (static_cast<size_t>(cf + c) + u) * 8 + h));
  // combine the 16 threads of the head
#pragma unroll
  for (int o = 8; o; o >>= 1) {
    const float Mo = __shfl_xor_sync(0xffffffffu, M, o), Lo = __shfl_xor_sync(0xffffffffu, L, o);
    const float Mn = fmaxf(M, Mo);
    L = (Mn == -INFINITY) ? 0.f : L * ex2(M - Mn) + Lo * ex2(Mo - Mn);
    M = Mn;
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int c = k + 16 * r;
    if (c < CH) wbuf[c * 8 + h] = (h < nh && c < nct) ? ex2(v[r].x - M) : 0.f;
  }
  for (int c = k + 64; c < min(nct, CH); c += 16)
    wbuf[c * 8 + h] = (h < nh) ? ex2(__ldcg(mlg + (static_cast<size_t>(cf + c) + u) * 8 + h).x - M) : 0.f;
  if (k == 0) {
    Mh[h] = M;
    Lh[h] = L;
  }
  named_bar_sync(1, 128);
  float4 acc[ITEMS];
#pragma unroll
  for (int i = 0; i < ITEMS; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (staged) {
    for (int b0 = 0, batch = 0; b0 < nct; b0 += NB, ++batch) {
      if (!mbar_wait(sbar, batch & 1)) *abort_flag = 1;
      named_bar_sync(1, 128);
      if (*abort_flag) {   // a copy that did not land in time: every thread leaves together
        if (tid == 0) atomicOr(p.err, FA_DEV_ERR_TIMEOUT);
        return;
      }
      const int n = min(NB, nct - b0);
      for (int c = 0; c < n; ++c) {
        const float* src = reinterpret_cast<const float*>(stage + c * ROW_BYTES);
#pragma unroll
        for (int i = 0; i < ITEMS; ++i) {
          const int idx = tid + i * 128, hh = idx / (D / 4), d = (idx % (D / 4)) * 4;
          const float w = wbuf[(b0 + c) * 8 + hh];
          const float4 o = *reinterpret_cast<const float4*>(src + hh * D + d);
          acc[i].x += w * o.x;
          acc[i].y += w * o.y;
          acc[i].z += w * o.z;
          acc[i].w += w * o.w;
        }
      }
      fence_proxy_async_smem();   // these generic reads before the next batch's bulk copies
      named_bar_sync(1, 128);     // every thread is done with this batch's rows
      if (b0 + NB < nct && tid == 0) stage_batch(b0 + NB, batch + 1);
    }
  }
  for (int c0 = 0; !staged && c0 < nct; c0 += CH) {
    const int n = min(CH, nct - c0);
    if (c0 > 0) {   // weights of later chunks (more than CH source CTAs)
      named_bar_sync(1, 128);
      for (int e = tid; e < n * 8; e += 128) {
        const int c = e >> 3, hh = e & 7;
        const float m = __ldcg(p.ml_part + (static_cast<size_t>(cf + c0 + c) + u) * 16 + hh * 2);
        wbuf[e] = (hh < nh) ? ex2(m - Mh[hh]) : 0.f;
      }
      named_bar_sync(1, 128);
    }
    // source CTAs outer, this thread's outputs inner: every iteration has
    // ITEMS independent L2 loads in flight
#pragma unroll 8
    for (int c = 0; c < n; ++c) {
      const float* src = p.o_part + (static_cast<size_t>(cf + c0 + c) + u) * 8 * D;
      float4 o[ITEMS];
#pragma unroll
      for (int i = 0; i < ITEMS; ++i) {
        const int idx = tid + i * 128, hh = idx / (D / 4), d = (idx % (D / 4)) * 4;
        o[i] = (hh < nh) ? __ldcg(reinterpret_cast<const float4*>(src + hh * D + d)) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int i = 0; i < ITEMS; ++i) {
        const float w = wbuf[c * 8 + (tid + i * 128) / (D / 4)];
        acc[i].x += w * o[i].x;
        acc[i].y += w * o[i].y;
        acc[i].z += w * o[i].z;
        acc[i].w += w * o[i].w;
      }
    }
  }
#pragma unroll
  for (int i = 0; i < ITEMS; ++i) {
    const int idx = tid + i * 128, hh = idx / (D / 4), d = (idx % (D / 4)) * 4;
    if (hh >= nh) continue;
    const float inv = Lh[hh] > 0.f ? 1.0f / Lh[hh] : 0.f;
    uint2 packed;
    packed.x = pack_bf16x2(acc[i].x * inv, acc[i].y * inv);
    packed.y = pack_bf16x2(acc[i].z * inv, acc[i].w * inv);
    *reinterpret_cast<uint2*>(p.out + (static_cast<size_t>(x.b) * p.Hq + head0 + hh) * D + d) = packed;
  }
  if (p.lse && tid < nh)
    p.lse[static_cast<size_t>(x.b) * p.Hq + head0 + tid] = (Mh[tid] + __log2f(Lh[tid])) * 0.69314718055994531f;
  named_bar_sync(1, 128);   // the scratch (the score-exchange buffer) is free again
}

// One CTA of a layer's decode: CTA `cta` of the `grid` CTAs launched for the
// layer (a launch may hold several layers; see decode_layers_kernel).
template <int D, int KV>
__device__ __forceinline__ void decode_body(const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                            const CUtensorMap* tm_ks, const CUtensorMap* tm_vs, const DecK& p,
                                            const int cta, const int grid) {
  using C = DecCfg<D, KV>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* sx = reinterpret_cast<float*>(smem + C::OFF_SX);
  __nv_bfloat16* qbuf = reinterpret_cast<__nv_bfloat16*>(smem + C::OFF_Q);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + C::NSTAGE;
  uint64_t* qfull = empty + C::NSTAGE;
  uint64_t* qempty = qfull + 1;
  uint64_t* mbar_merge = qempty + 1;
  __shared__ int sm_scan[8], sm_mm[16];
  __shared__ int sh_u0, sh_p0, sh_n0, abort_flag, sh_last;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;

  // Inputs may come from the previous kernel in the stream.  With early
  // metadata the caller guarantees that kernel writes no block table or
  // sequence length, so the partition below (and the first page ids) may be
  // read before waiting for it; q, the slabs and the outputs always wait.
  if (!p.early_metadata) griddep_wait();
  griddep_launch_dependents();

  // ---------------------------------------------------------------- partition
  // One block scan gives every unit's first global tile P_u and the total T.
  // Two ways to cut the tile lists into CTA shares:
  //  * unit-aligned: when every unit has about the same number of tiles (the
  //    sliding layers once L >= W), each unit is cut into kper equal parts,
  //    one CTA each, so no CTA crosses a unit boundary and every merge has
  //    exactly kper partials;
  //  * concatenated: otherwise the lists are laid end to end and cut into
  //    ncta equal shares, so every CTA moves the same bytes whatever the
  //    length mix.
  int T = 0, my_n = 0, my_P = 0;
  {
    int running = 0;
    for (int base = 0; base < p.units; base += blockDim.x) {
      const int u = base + threadIdx.x;
      Unit x{};
      if (u < p.units) {
        x = unit_of(p, u);
        if (cta == 0 && __ldg(p.seq_lens + x.b) > p.max_seq_len) atomicOr(p.err, FA_DEV_ERR_BOUND);
      }
      int tot;
      const int P = running + block_excl_scan(x.n, sm_scan, &tot);
      if (base == 0) {
        my_n = x.n;
        my_P = P;
      }
      running += tot;
    }
    T = running;
  }
  int ncta = (T == 0) ? 0 : min(grid, max(1, (T + p.min_tiles - 1) / p.min_tiles));
  int kper = 0;   // CTAs per unit of the unit-aligned cut (0: concatenated cut)
  if (ncta > 0 && p.units <= static_cast<int>(blockDim.x)) {
    const bool mine = static_cast<int>(threadIdx.x) < p.units;
    const int2 r = block_min_max(mine ? my_n : INT_MAX, mine ? my_n : 0, sm_mm);
    if (r.x >= 1 && r.y - r.x <= max(1, r.x >> 3)) {
      const int k = min(ncta / p.units, r.x);
      // take it only if it keeps at least 85% of the concatenated cut's CTAs
      if (k >= 1 && 20 * k * p.units >= 17 * ncta) {
        kper = k;
        ncta = k * p.units;
      }
    }
  }
  if (cta >= ncta) {
    if (ncta == 0 && cta == 0) {   // nothing visible anywhere: only empty outputs to write
      griddep_wait();
      zero_empty_units<D, KV>(p, 0, 1, threadIdx.x, blockDim.x);
    }
    return;
  }
  long long s_beg = static_cast<long long>(cta) * T / ncta;
  long long s_end = static_cast<long long>(cta + 1) * T / ncta;
  if (kper) {
    if (static_cast<int>(threadIdx.x) == cta / kper) {
      sh_u0 = threadIdx.x;
      sh_p0 = my_P;
      sh_n0 = my_n;
    }
  } else if (p.units <= static_cast<int>(blockDim.x)) {
    if (my_n > 0 && my_P <= s_beg && s_beg < my_P + my_n) {
      sh_u0 = threadIdx.x;
      sh_p0 = my_P;
    }
  } else {
    int running = 0;
    for (int base = 0; base < p.units; base += blockDim.x) {
      const int u = base + threadIdx.x;
      const int n = (u < p.units) ? unit_of(p, u).n : 0;
      int tot;
      const int P = running + block_excl_scan(n, sm_scan, &tot);
      if (n > 0 && P <= s_beg && s_beg < P + n) {
        sh_u0 = u;
        sh_p0 = P;
      }
      running += tot;
    }
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NSTAGE; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C::NCW);
    }
    mbar_init(qfull, 1);
    mbar_init(qempty, C::NCW);
    mbar_init(mbar_merge, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const int u0 = sh_u0, p0 = sh_p0;
  if (kper) {   // part r of unit u0
    const int r = cta % kper, n0 = sh_n0;
    s_beg = p0 + static_cast<long long>(r) * n0 / kper;
    s_end = p0 + static_cast<long long>(r + 1) * n0 / kper;
  }

  if (warp == C::NCW) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(tm_k);
      prefetch_tmap(tm_v);
    }
    const uint64_t pol = l2_policy_evict_first();
    int gi = 0, j = 0;
    bool ok = true;
    long long P = p0;
    for (int u = u0; ok && P < s_end; ++u) {
      const Unit x = unit_of(p, u);
      if (x.n > 0) {
        const int ta = x.t_first + static_cast<int>(max(s_beg, P) - P);
        const int tz = x.t_first + static_cast<int>(min(s_end, P + x.n) - P);
        const int nh = min(8, p.g - x.c * 8), head0 = x.h * p.g + x.c * 8;
        const int32_t* bt = p.block_table + static_cast<size_t>(x.b) * p.max_pages_per_seq;
        // The CTA that reads the unit's last tile (it holds position L - 1)
        // stores the current token's rows first, so its own copy of that
        // tile sees them.
        const bool store_here = p.slots != nullptr && tz == x.t_first + x.n;
        bool stored = false;
        RowRegs<D> rk, rv;
        for (int k0 = ta; ok && k0 < tz; k0 += 32) {
          int pid = -1;
          if (k0 + lane < tz) {
            pid = __ldg(bt + (k0 + lane) / p.tiles_per_page);
            if (pid < 0 || pid >= p.num_pages) {
              atomicOr(p.err, FA_DEV_ERR_PAGE);
              pid = -1;   // the TMA box then lies outside the tensor and reads zeros
            }
          }
          if (k0 == ta) {
            if (j == 0 && p.early_metadata && k0 + lane < tz && lane < C::PREFETCH_TILES && pid >= 0) {
              // While the preceding kernel finishes, pull this CTA's first
              // tiles into L2.  A prefetch returns nothing to the SM, so it is
              // safe even if that kernel is still writing the slab; the TMA
              // loads below read only after the dependency resolves.
              const size_t row0 = (static_cast<size_t>(pid) * p.Hkv + x.h) * p.page_size +
                                  ((k0 + lane) % p.tiles_per_page) * kTile;
              prefetch_l2(p.kb + row0 * C::ROWB, C::TILE_BYTES);
              prefetch_l2(p.vb + row0 * C::ROWB, C::TILE_BYTES);
              if constexpr (KV) {
                prefetch_l2(p.ksb + row0, kTile * sizeof(float));
                prefetch_l2(p.vsb + row0, kTile * sizeof(float));
              }
            }
            if (j == 0) griddep_wait();   // from here on q and the slab are read
            if (lane == 0) {
              if (j > 0) ok = mbar_wait(qempty, (j - 1) & 1);
              if (ok) {
                mbar_arrive_expect_tx(qfull, nh * D * 2);
                bulk_load(qbuf, p.q + (static_cast<size_t>(x.b) * p.Hq + head0) * D, nh * D * 2, qfull);
              }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            if (store_here) {   // issue the row loads now; they are written before the last tile's copy
              const size_t src = (static_cast<size_t>(x.b) * p.Hkv + x.h) * D;
              row_load<D>(rk, p.k_new + src, lane);
              row_load<D>(rv, p.v_new + src, lane);
            }
          }
          for (int k = k0; k < min(k0 + 32, tz); k += C::NT) {
            const int ntl = min(C::NT, tz - k);
            if (store_here && !stored && k + ntl >= tz) {
              stored = true;
              store_current<D, KV>(p, rk, rv, x.h, __ldg(p.slots + x.b), lane);
              // each lane orders its generic writes before the async-proxy
              // (TMA) read of the tile that holds them
              fence_proxy_async_global();
              __syncwarp();
            }
            int pg[C::NT];
#pragma unroll
            for (int t = 0; t < C::NT; ++t) pg[t] = __shfl_sync(0xffffffffu, pid, (k - k0 + t) & 31);
            if (lane == 0) {
              const int st = gi % C::NSTAGE;
              ok = mbar_wait(&empty[st], ((gi / C::NSTAGE) & 1) ^ 1);
              if (ok) {
                mbar_arrive_expect_tx(&full[st], ntl * (2 * C::TILE_BYTES + (KV ? 128 : 0)));
                uint8_t* kdst = smem + st * C::STAGE_KV;
                uint8_t* vdst = kdst + C::NT * C::TILE_BYTES;
                for (int t = 0; t < ntl; ++t) {
                  const int tile = k + t;
                  const int row0 = (pg[t] * p.Hkv + x.h) * p.page_size + (tile % p.tiles_per_page) * kTile;
                  // one copy per tile: all column blocks of 16 rows
                  tma_load_3d(kdst + t * C::TILE_BYTES, tm_k, &full[st], 0, row0, 0, pol);
                  tma_load_3d(vdst + t * C::TILE_BYTES, tm_v, &full[st], 0, row0, 0, pol);
                  if constexpr (KV) {
                    float* sc = reinterpret_cast<float*>(smem + C::OFF_SC + st * C::SC_BYTES);
                    tma_load_2d(sc + t * 32, tm_ks, &full[st], 0, row0 / kTile, pol);
                    tma_load_2d(sc + (C::NT + t) * 32, tm_vs, &full[st], 0, row0 / kTile, pol);
                  }
                }
              }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            ++gi;
          }
        }
        ++j;
      }
      P += x.n;
    }
    if (lane == 0) {
      if (!ok) atomicOr(p.err, FA_DEV_ERR_TIMEOUT);
      // drain: no bulk copy may still be landing when the CTA exits
      for (int i = max(0, gi - C::NSTAGE); i < gi; ++i)
        if (!mbar_wait(&full[i % C::NSTAGE], (i / C::NSTAGE) & 1)) atomicOr(p.err, FA_DEV_ERR_TIMEOUT);
      if (j > 0 && !mbar_wait(qfull, (j - 1) & 1)) atomicOr(p.err, FA_DEV_ERR_TIMEOUT);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  griddep_wait();
  zero_empty_units<D, KV>(p, cta, ncta, threadIdx.x, C::NCW * 32);
  const int qk_tile = warp % C::NT;
  const int qk_d0 = (warp / C::NT) * C::QK_COLS;
  const int pv_d0 = warp * C::PV_COLS;
  constexpr int QF = KV ? C::QK_COLS / 32 : C::QK_COLS / 16;
  int gi = 0, j = 0;
  long long P = p0;
  for (int u = u0; P < s_end; ++u) {
    const Unit x = unit_of(p, u);
    if (x.n == 0) continue;   // an empty unit advances nothing
    const int ta = x.t_first + static_cast<int>(max(s_beg, P) - P);
    const int tz = x.t_first + static_cast<int>(min(s_end, P + x.n) - P);
    const int nh = min(8, p.g - x.c * 8), head0 = x.h * p.g + x.c * 8;
    const int qpos = x.L - 1, lo = x.lo;
    const bool hv = gid < nh;

    // queries of this segment: Q^T fragments (B operand), zero for padded heads
    // every wait below is made warp-uniform (and the warp reconverged) by a
    // vote, since ldmatrix and mma.sync need all 32 lanes together
    const bool qok = __all_sync(0xffffffffu, mbar_wait(qfull, j & 1));
    if (!qok && lane == 0) {
      abort_flag = 1;
      atomicOr(p.err, FA_DEV_ERR_TIMEOUT);
    }
    uint32_t qf[QF][KV ? 4 : 2];
    {
      uint32_t qbig = 0;   // 8-bit formats: a query element f16 cannot hold
      const __nv_bfloat16* qrow = qbuf + (hv ? gid : 0) * D;
#pragma unroll
      for (int kk = 0; kk < QF; ++kk) {
        if constexpr (!KV) {
          const int d = qk_d0 + kk * 16 + 2 * tig;
          qf[kk][0] = hv ? *reinterpret_cast<const uint32_t*>(qrow + d) : 0u;
          qf[kk][1] = hv ? *reinterpret_cast<const uint32_t*>(qrow + d + 8) : 0u;
        } else {
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const int d = qk_d0 + kk * 32 + half * 16 + 4 * tig;
            const uint2 w = hv ? *reinterpret_cast<const uint2*>(qrow + d) : make_uint2(0u, 0u);
            qbig |= bf16x2_past_f16(w.x) | bf16x2_past_f16(w.y);
            qf[kk][2 * half + 0] = pack_f16x2_sat(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u));
            qf[kk][2 * half + 1] = pack_f16x2_sat(__uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
          }
        }
      }
      if constexpr (KV != 0) {
        if (__any_sync(0xffffffffu, qbig != 0) && lane == 0) atomicOr(p.err, FA_DEV_ERR_RANGE);
      }
    }
    // qbuf is refilled by a bulk copy (async proxy) once every warp has
    // arrived: each thread's generic reads of it are ordered before that
    // write by a proxy fence, which also waits for loads still in flight
    // (the fragments are not used before the arrive)
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(qempty);

    float o[C::PV_MT][4];
#pragma unroll
    for (int i = 0; i < C::PV_MT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
    float m_run = -INFINITY, l_run = 0.0f, sigma = 1.0f;

    for (int tile0 = ta; tile0 < tz; tile0 += C::NT) {
      const int st = gi % C::NSTAGE;
      const int buf = gi & 1;
      const int ntl = min(C::NT, tz - tile0);
      const uint8_t* ks = smem + st * C::STAGE_KV;
      const uint8_t* vs = ks + C::NT * C::TILE_BYTES;
      const float* scl = reinterpret_cast<const float*>(smem + C::OFF_SC + st * C::SC_BYTES);
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&full[st], (gi / C::NSTAGE) & 1));
      if (!ok && lane == 0) {
        abort_flag = 1;
        atomicOr(p.err, FA_DEV_ERR_TIMEOUT);
      }

      // ---- partial S^T over this warp's columns
      // two accumulator chains (even / odd column steps) halve the dependent MMA chain
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      float acc1[4] = {0.f, 0.f, 0.f, 0.f};
      if (ok && qk_tile < ntl) {
        const uint8_t* kt = ks + qk_tile * C::TILE_BYTES;
        const int r = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
        for (int kk = 0; kk < QF; ++kk) {
          uint32_t a0, a1, a2, a3;
          if constexpr (!KV) {
            const int dc = qk_d0 + kk * 16 + (lane >> 4) * 8;
            ldsm_x4(smem_u32(kt + (dc >> 6) * 2048 + sw128(r, (dc & 63) >> 3)), a0, a1, a2, a3);
            mma_bf16((kk & 1) ? acc1 : acc, a0, a1, a2, a3, qf[kk][0], qf[kk][1]);
          } else {
            const int dc = qk_d0 + kk * 32 + (lane >> 4) * 16;
            ldsm_x4(smem_u32(kt + (dc >> 7) * 2048 + sw128(r, (dc & 127) >> 4)), a0, a1, a2, a3);
            mma_f16(acc, codes_to_f16x2<KV, 0, 1>(a0), codes_to_f16x2<KV, 0, 1>(a1), codes_to_f16x2<KV, 2, 3>(a0),
                    codes_to_f16x2<KV, 2, 3>(a1), qf[kk][0], qf[kk][1]);
            mma_f16(acc1, codes_to_f16x2<KV, 0, 1>(a2), codes_to_f16x2<KV, 0, 1>(a3), codes_to_f16x2<KV, 2, 3>(a2),
                    codes_to_f16x2<KV, 2, 3>(a3), qf[kk][2], qf[kk][3]);
          }
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[i] += acc1[i];
      float* sxw = sx + (buf * C::NCW + warp) * kTile * C::SX_STRIDE;
      *reinterpret_cast<float2*>(sxw + gid * C::SX_STRIDE + 2 * tig) = make_float2(acc[0], acc[1]);
      *reinterpret_cast<float2*>(sxw + (gid + 8) * C::SX_STRIDE + 2 * tig) = make_float2(acc[2], acc[3]);
      named_bar_sync(1, C::NCW * 32);
      if (*reinterpret_cast<volatile int*>(&abort_flag)) goto consumers_done;

      {
        // ---- scores for this lane's head (gid), keys {2tig, 2tig+1, 2tig+8, 2tig+9} of each tile
        float s[C::NT][4];
        bool valid[C::NT][4];
        float mloc = -INFINITY;
#pragma unroll
        for (int t = 0; t < C::NT; ++t) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int key = 2 * tig + (e & 1) + (e >> 1) * 8;
            float v = 0.0f;
#pragma unroll
            for (int w = t; w < C::NCW; w += C::NT) v += sx[((buf * C::NCW + w) * kTile + key) * C::SX_STRIDE + gid];
            const int pos = (tile0 + t) * kTile + key;
            valid[t][e] = (t < ntl) && pos >= lo && pos <= qpos;
            float sc = p.scale_log2;
            if constexpr (KV) sc *= scl[t * 32 + key];
            s[t][e] = valid[t][e] ? v * sc : -INFINITY;
            mloc = fmaxf(mloc, s[t][e]);
          }
        }
        mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 1));
        mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 2));
        const float m_new = fmaxf(m_run, mloc);
        const float alpha = (m_run == -INFINITY) ? 0.0f : ex2(m_run - m_new);
        float psum = 0.0f;
        uint32_t pf[C::NT][2];
        float vmax = 1.0f, ivm = 1.0f;
        float vsc[C::NT][4];   // 8-bit: this lane's keys' V scales (0 where not visible)
        if constexpr (KV) {
          float vm = 0.0f;
#pragma unroll
          for (int t = 0; t < C::NT; ++t)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              vsc[t][e] = valid[t][e] ? scl[(C::NT + t) * 32 + 2 * tig + (e & 1) + (e >> 1) * 8] : 0.0f;
              vm = fmaxf(vm, vsc[t][e]);
            }
          vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, 1));
          vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, 2));
          vmax = vm > 0.0f ? vm : 1.0f;
          ivm = __frcp_rn(vmax);   // one reciprocal per step instead of a division per weight
        }
#pragma unroll
        for (int t = 0; t < C::NT; ++t) {
          float pe[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            pe[e] = ex2(s[t][e] - m_new);
            if constexpr (KV) {
              psum += pe[e];
              pe[e] *= vsc[t][e] * ivm;
            }
          }
          if constexpr (!KV) {
            // the denominator sums the bf16-rounded weights the PV MMA uses, so
            // the weights of each output row sum to exactly one
            pf[t][0] = pack_bf16x2(pe[0], pe[1]);
            pf[t][1] = pack_bf16x2(pe[2], pe[3]);
            psum += __uint_as_float(pf[t][0] << 16) + __uint_as_float(pf[t][0] & 0xffff0000u) +
                    __uint_as_float(pf[t][1] << 16) + __uint_as_float(pf[t][1] & 0xffff0000u);
          } else {
            pf[t][0] = pack_f16x2(pe[0], pe[1]);
            pf[t][1] = pack_f16x2(pe[2], pe[3]);
          }
        }
        l_run = l_run * alpha + psum;
        m_run = m_new;
        float ofac = alpha;
        if constexpr (KV) {
          ofac = alpha * sigma * ivm;
          sigma = vmax;
        }
        // rescale O: this lane's O columns are heads 2tig and 2tig+1
        const float fa_ = __shfl_sync(0xffffffffu, ofac, 8 * tig);
        const float fb_ = __shfl_sync(0xffffffffu, ofac, 8 * tig + 4);
#pragma unroll
        for (int mt = 0; mt < C::PV_MT; ++mt) {
          o[mt][0] *= fa_;
          o[mt][1] *= fb_;
          o[mt][2] *= fa_;
          o[mt][3] *= fb_;
        }

        if constexpr (KV != FA_KV_INT8) {
          // masked keys have p = 0, but their V rows may hold anything (NaN
          // included; e4m3 has NaN codes too, int8 has none): zero this
          // warp's columns of those rows before the MMA
          if (tile0 * kTile < lo || (tile0 + ntl) * kTile - 1 > qpos) {
            constexpr int EPU = 16 / C::ELEM;              // elements per 16-byte unit
            constexpr int UNITS = C::PV_COLS / EPU;        // 16-byte units per row slice
            constexpr int EPB = 128 / C::ELEM;             // elements per 128-byte column block
            uint8_t* vw = const_cast<uint8_t*>(vs);
            for (int t = 0; t < ntl; ++t) {
              for (int idx = lane; idx < kTile * UNITS; idx += 32) {
                const int r = idx / UNITS, uu = idx % UNITS;
                const int pos = (tile0 + t) * kTile + r;
                if (pos < lo || pos > qpos) {
                  const int dc = pv_d0 + uu * EPU;
                  *reinterpret_cast<uint4*>(vw + t * C::TILE_BYTES + (dc / EPB) * 2048 +
                                            sw128(r, (dc % EPB) / EPU)) = make_uint4(0u, 0u, 0u, 0u);
                }
              }
            }
            fence_proxy_async_smem();
            __syncwarp();
          }
        }

        // ---- O^T += V^T P^T over this warp's columns
#pragma unroll
        for (int t = 0; t < C::NT; ++t) {
          if (t >= ntl) break;
          const uint8_t* vt = vs + t * C::TILE_BYTES;
          const int r = (lane & 7) + (lane >> 4) * 8;
          if constexpr (!KV) {
#pragma unroll
            for (int mt = 0; mt < C::PV_MT; ++mt) {
              const int dc = pv_d0 + mt * 16 + ((lane >> 3) & 1) * 8;
              uint32_t a0, a1, a2, a3;
              ldsm_x4_t(smem_u32(vt + (dc >> 6) * 2048 + sw128(r, (dc & 63) >> 3)), a0, a1, a2, a3);
              mma_bf16(o[mt], a0, a1, a2, a3, pf[t][0], pf[t][1]);
            }
          } else {
#pragma unroll
            for (int gi2 = 0; gi2 < C::PV_MT / 2; ++gi2) {
              const int dc = pv_d0 + gi2 * 32 + ((lane >> 3) & 1) * 16;
              uint32_t r0, r1, r2, r3;
              ldsm_x4_t(smem_u32(vt + (dc >> 7) * 2048 + sw128(r, (dc & 127) >> 4)), r0, r1, r2, r3);
              mma_f16(o[2 * gi2], codes_to_f16x2<KV, 0, 2>(r0), codes_to_f16x2<KV, 0, 2>(r1),
                      codes_to_f16x2<KV, 0, 2>(r2), codes_to_f16x2<KV, 0, 2>(r3), pf[t][0], pf[t][1]);
              mma_f16(o[2 * gi2 + 1], codes_to_f16x2<KV, 1, 3>(r0), codes_to_f16x2<KV, 1, 3>(r1),
                      codes_to_f16x2<KV, 1, 3>(r2), codes_to_f16x2<KV, 1, 3>(r3), pf[t][0], pf[t][1]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
      ++gi;
    }

    {
      // ------------------------------------------------------ segment epilogue
      l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
      l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
      const int hA = 2 * tig, hB = 2 * tig + 1;
      const float lA = __shfl_sync(0xffffffffu, l_run, 8 * tig);
      const float lB = __shfl_sync(0xffffffffu, l_run, 8 * tig + 4);
      // output column d of C-fragment row (gid + 8 * half) of O^T tile mt
      auto out_d = [&](int mt, int half) -> int {
        if constexpr (!KV) return pv_d0 + mt * 16 + gid + 8 * half;
        else return pv_d0 + (mt >> 1) * 32 + 16 * half + 2 * gid + (mt & 1);
      };
      const int c_first = kper ? u * kper : cta_of(P, ncta, T);
      const int c_last = kper ? c_first + kper - 1 : cta_of(P + x.n - 1, ncta, T);
      if (c_first == c_last) {
        const float iA = (lA > 0.f) ? sigma / lA : 0.f, iB = (lB > 0.f) ? sigma / lB : 0.f;
#pragma unroll
        for (int mt = 0; mt < C::PV_MT; ++mt)
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const int d = out_d(mt, half);
            if (hA < nh)
              p.out[(static_cast<size_t>(x.b) * p.Hq + head0 + hA) * D + d] = __float2bfloat16_rn(o[mt][2 * half] * iA);
            if (hB < nh)
              p.out[(static_cast<size_t>(x.b) * p.Hq + head0 + hB) * D + d] =
                  __float2bfloat16_rn(o[mt][2 * half + 1] * iB);
          }
        if (p.lse && warp == 0 && tig == 0 && hv)
          p.lse[static_cast<size_t>(x.b) * p.Hq + head0 + gid] = (m_run + __log2f(l_run)) * 0.69314718055994531f;
      } else {
        const size_t slot = static_cast<size_t>(cta) + u;
#pragma unroll
        for (int mt = 0; mt < C::PV_MT; ++mt)
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const int d = out_d(mt, half);
            p.o_part[(slot * 8 + hA) * D + d] = o[mt][2 * half] * sigma;
            p.o_part[(slot * 8 + hB) * D + d] = o[mt][2 * half + 1] * sigma;
          }
        if (warp == 0 && tig == 0)
          reinterpret_cast<float2*>(p.ml_part)[slot * 8 + gid] = make_float2(m_run, l_run);
        // arrive; the last of the unit's CTAs merges every partial row.  The
        // barrier orders the CTA's partial writes before thread 0's
        // release/acquire add, which publishes them and, for the last
        // arrival, makes the other CTAs' rows visible.
        named_bar_sync(1, C::NCW * 32);
        if (threadIdx.x == 0) {
          const int nct = c_last - c_first + 1;
          const int old = atom_add_acq_rel_gpu(p.counters + u, 1);
          int last = 0;
          if (old == nct - 1) {
            last = 1;
            atomicExch(p.counters + u, 0);   // leave the counter zero for the next call
          } else if (old >= nct) {
            atomicOr(p.err, FA_DEV_ERR_WORKSPACE);
          }
          sh_last = last;
        }
        named_bar_sync(1, C::NCW * 32);
        if (sh_last) {
          // the ring is idle once this CTA's last segment is consumed: stage the merge there
          const bool idle = P + x.n >= s_end;
          merge_unit<D, C::STAGE_ALL>(p, u, x, nh, head0, c_first, c_last, sx, idle ? smem : nullptr, mbar_merge,
                                       &abort_flag);
        }
      }
    }
    ++j;
    P += x.n;
  }
consumers_done:;
}

template <int D, int KV>
__global__ void __launch_bounds__(DecCfg<D, KV>::NTHR, 2)
    decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_ks, const __grid_constant__ CUtensorMap tm_vs,
                  const DecK p) {
  decode_body<D, KV>(&tm_k, &tm_v, &tm_ks, &tm_vs, p, static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x));
}

// Several layers of one head_dim and KV format in one launch: the CTAs of
// layer i are [cta0[i], cta0[i + 1]); each runs exactly as in a launch of
// its own, with its own parameters, tensor maps and workspace region.
struct DecLayers {
  CUtensorMap tm[kMaxLayersPerLaunch][4];   // K, V, K scale, V scale
  DecK k[kMaxLayersPerLaunch];
  int cta0[kMaxLayersPerLaunch + 1];
  int n;
};

template <int D, int KV>
__global__ void __launch_bounds__(DecCfg<D, KV>::NTHR, 2) decode_layers_kernel(const __grid_constant__ DecLayers m) {
  const int b = static_cast<int>(blockIdx.x);
  int li = 0;
  while (li + 1 < m.n && b >= m.cta0[li + 1]) ++li;
  decode_body<D, KV>(&m.tm[li][0], &m.tm[li][1], &m.tm[li][2], &m.tm[li][3], m.k[li], b - m.cta0[li],
                     m.cta0[li + 1] - m.cta0[li]);
}

template <int D, int KV>
static cudaError_t launch_decode_t(const DecodeArgs& a, const DecK& k, cudaStream_t s) {
  using C = DecCfg<D, KV>;
  static unsigned int done = 0;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(decode_kernel<D, KV>), C::SMEM_ALLOC, &done);
  if (e != cudaSuccess) return e;
  e = launch_pdl(decode_kernel<D, KV>, dim3(a.plan.ncta), dim3(C::NTHR), C::SMEM_ALLOC, s, *a.tm_k, *a.tm_v,
                 *a.tm_ks, *a.tm_vs, k);
  return e;
}

template <int D, int KV>
static cudaError_t launch_decode_layers_t(const DecLayers& m, cudaStream_t s) {
  using C = DecCfg<D, KV>;
  static unsigned int done = 0;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(decode_layers_kernel<D, KV>), C::SMEM_ALLOC, &done);
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_layers_kernel<D, KV>, dim3(m.cta0[m.n]), dim3(C::NTHR), C::SMEM_ALLOC, s, m);
}

// The kernel parameters of one layer's decode.
static DecK make_deck(const DecodeArgs& a) {
  DecK k{};
  k.q = static_cast<const __nv_bfloat16*>(a.q);
  k.block_table = a.block_table;
  k.seq_lens = a.seq_lens;
  k.kb = static_cast<uint8_t*>(const_cast<void*>(a.k));
  k.vb = static_cast<uint8_t*>(const_cast<void*>(a.v));
  k.ksb = const_cast<float*>(a.k_scale);
  k.vsb = const_cast<float*>(a.v_scale);
  k.k_new = static_cast<const __nv_bfloat16*>(a.k_new);
  k.v_new = static_cast<const __nv_bfloat16*>(a.v_new);
  k.slots = a.slots;
  k.out = static_cast<__nv_bfloat16*>(a.out);
  k.lse = a.lse;
  if (a.workspace) {
    char* ws = static_cast<char*>(a.workspace);
    k.counters = reinterpret_cast<int*>(ws);
    k.ml_part = reinterpret_cast<float*>(ws + a.plan.off_ml);
    k.o_part = reinterpret_cast<float*>(ws + a.plan.off_o);
  }
  k.err = a.err;
  k.B = a.B;
  k.Hq = a.Hq;
  k.Hkv = a.Hkv;
  k.g = a.Hq / a.Hkv;
  k.chunks = a.plan.head_chunks;
  k.kind = a.kind;
  k.window = a.window;
  k.page_size = a.page_size;
  k.tiles_per_page = a.page_size / kTile;
  k.num_pages = a.num_pages;
  k.max_pages_per_seq = a.max_pages_per_seq;
  k.max_seq_len = a.max_seq_len;
  k.units = a.plan.units;
  k.min_tiles = a.plan.min_tiles;
  k.early_metadata = a.early_metadata;
  k.scale_log2 = a.sm_scale * 1.4426950408889634f;
  return k;
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
  const DecK k = make_deck(a);
  if (a.kv_dtype == FA_KV_INT8) {
    if (a.D == 256) return launch_decode_t<256, FA_KV_INT8>(a, k, s);
    return launch_decode_t<512, FA_KV_INT8>(a, k, s);
  }
  if (a.kv_dtype == FA_KV_FP8) {
    if (a.D == 256) return launch_decode_t<256, FA_KV_FP8>(a, k, s);
    return launch_decode_t<512, FA_KV_FP8>(a, k, s);
  }
  if (a.D == 256) return launch_decode_t<256, FA_KV_BF16>(a, k, s);
  return launch_decode_t<512, FA_KV_BF16>(a, k, s);
}

cudaError_t launch_decode_layers(const DecodeArgs* a, int n, cudaStream_t s) {
  if (n < 1 || n > kMaxLayersPerLaunch) return cudaErrorInvalidValue;
  DecLayers m{};   // the kernel parameters (copied at launch)
  m.n = n;
  m.cta0[0] = 0;
  for (int i = 0; i < n; ++i) {
    m.tm[i][0] = *a[i].tm_k;
    m.tm[i][1] = *a[i].tm_v;
    m.tm[i][2] = *a[i].tm_ks;
    m.tm[i][3] = *a[i].tm_vs;
    m.k[i] = make_deck(a[i]);
    m.cta0[i + 1] = m.cta0[i] + a[i].plan.ncta;
  }
  if (a[0].kv_dtype == FA_KV_INT8) {
    if (a[0].D == 256) return launch_decode_layers_t<256, FA_KV_INT8>(m, s);
    return launch_decode_layers_t<512, FA_KV_INT8>(m, s);
  }
  if (a[0].kv_dtype == FA_KV_FP8) {
    if (a[0].D == 256) return launch_decode_layers_t<256, FA_KV_FP8>(m, s);
    return launch_decode_layers_t<512, FA_KV_FP8>(m, s);
  }
  if (a[0].D == 256) return launch_decode_layers_t<256, FA_KV_BF16>(m, s);
  return launch_decode_layers_t<512, FA_KV_BF16>(m, s);
}

// ---------------------------------------------------------------------------
// Allocation-free decode: the same kernel with its scratch in a file-scope
// device array of FA_NOALLOC_SCRATCH_BYTES, for callers that cannot allocate
// device memory.  The array is part of the loaded module, so every GPU that
// loads the library holds it until the process exits.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, never a device address, so
// the address is looked up once per device (with that device current).
static void* noalloc_scratch(cudaError_t* err) {
  static std::mutex mu;
  static void* ptrs[128] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 128) {
    *err = e != cudaSuccess ? e : cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) {
      *err = e;
      return nullptr;
    }
    ptrs[dev] = p;
  }
  *err = cudaSuccess;
  return ptrs[dev];
}

}  // namespace fa

extern "C" fa_status fa_paged_decode_attn_noalloc(fa_cache* cache, int32_t layer, const void* q,
                                                  const int32_t* block_table, int32_t max_pages_per_seq,
                                                  const int32_t* seq_lens, int32_t B, int32_t max_seq_len,
                                                  void* out, float* lse, void* stream) {
  if (!cache || layer < 0 || layer >= static_cast<int32_t>(cache->layers.size()))
    return fa::fail(FA_ERR_INVALID_ARG, "cache is NULL or layer %d out of range", layer);
  if (B <= 0 || max_seq_len <= 0)   // let the regular entry point validate and report
    return fa_paged_decode_attn(cache, layer, q, block_table, max_pages_per_seq, seq_lens, B, max_seq_len, out,
                                lse, nullptr, 0, stream);
  const fa::DecodePlan plan = fa::plan_decode(cache, layer, B, max_seq_len);
  if (plan.ws_bytes > FA_NOALLOC_SCRATCH_BYTES)
    return fa::fail(FA_ERR_WORKSPACE,
                    "allocation-free decode needs %zu bytes of scratch for B=%d, max_seq_len=%d; its fixed "
                    "scratch holds %zu bytes (use fa_paged_decode_attn with a caller workspace)",
                    plan.ws_bytes, B, max_seq_len, static_cast<size_t>(FA_NOALLOC_SCRATCH_BYTES));
  void* ws = nullptr;
  if (plan.ws_bytes) {
    cudaError_t ce;
    ws = fa::noalloc_scratch(&ce);
    if (!ws) return fa::fail(FA_ERR_CUDA, "scratch address lookup: %s", cudaGetErrorString(ce));
    // the arrival counters must start at zero whatever an earlier call left
    ce = cudaMemsetAsync(ws, 0, plan.off_ml, static_cast<cudaStream_t>(stream));
    if (ce != cudaSuccess) return fa::fail(FA_ERR_CUDA, "clearing scratch counters: %s", cudaGetErrorString(ce));
  }
  return fa_paged_decode_attn(cache, layer, q, block_table, max_pages_per_seq, seq_lens, B, max_seq_len, out, lse,
                              ws, plan.ws_bytes, stream);
}
