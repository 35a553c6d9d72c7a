// Paged decode attention: split-K online softmax, GQA-packed.
//
// Regimes ("unsloth gemma4_flex_inference.py" history, commit "block mask per
// attention regime"; "pegainfer issue #807", Description): a full layer's
// query at q_pos = L - 1 sees keys [0, q_pos]; a sliding layer's sees
// [max(0, L - W), q_pos].  Sliding layers only visit the 16-row tiles that
// hold in-window keys.  KV-shared layers arrive here with their source's slab
// ("FreeToken PR #898", description).
//
// Work decomposition.  grid = (split, KV head x head chunk, sequence).  One CTA
// walks `tiles_per_split` 16-row tiles of one sequence and one KV head and
// serves up to 8 query heads of that KV head at once, so each KV byte is read
// from HBM once for the whole group.  Per tile the contraction is
//   S^T (16 keys x 8 heads)  = K (16 x D) . Q^T (D x 8)         (mma.sync m16n8k16)
//   O^T (D x 8 heads)       += V^T (D x 16) . P^T (16 x 8)
// with keys on the MMA M side, so 8 heads fill N exactly.  Warp 4 is a TMA
// producer: it streams K and V tiles (and int8 scales) into a 3-stage ring of
// 128-byte-swizzled shared-memory tiles.  Warps 0-3 split the QK^T
// contraction over columns, exchange partial scores through shared memory,
// run the online softmax redundantly (each lane owns one head) and each
// accumulates its own quarter of O's columns.
//
// bf16 slabs use bf16 MMAs.  int8 slabs: codes become exact fp16 integers
// (byte permute + one subtraction), the K scale multiplies the fp32 scores,
// the V scale is folded into P (normalised by the step's largest scale, which
// joins the running rescale), and the MMAs run in fp16.
#include <cfloat>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {

template <int D, int KV>
struct DecCfg {
  static constexpr int ELEM = KV ? 1 : 2;
  static constexpr int ROWB = D * ELEM;                 // bytes per row
  static constexpr int NBLK = ROWB / 128;               // 128-byte column blocks per row
  static constexpr int TILE_BYTES = kTile * ROWB;       // one 16-row tile of K (or V)
  static constexpr int NT = 32768 / (2 * TILE_BYTES);   // tiles per pipeline step (32 KB of K+V)
  static constexpr int NSTAGE = 3;
  static constexpr int NCW = 4;                         // consumer warps
  static constexpr int QK_COLS = D * NT / NCW;          // QK^T columns per warp
  static constexpr int PV_COLS = D / NCW;               // output columns per warp
  static constexpr int PV_MT = PV_COLS / 16;            // m16 tiles of O^T per warp
  static constexpr int STAGE_KV = 2 * NT * TILE_BYTES;
  static constexpr int SC_BYTES = KV ? 2 * NT * 128 : 0; // k, v scales of the step's tiles (128-B slots)
  static constexpr int SX_STRIDE = 12;                  // floats per key row (bank-conflict free)
  static constexpr int SX_BYTES = 2 * NCW * kTile * SX_STRIDE * 4;
  static constexpr int MAX_TPS = 512;
  static constexpr int OFF_SC = NSTAGE * STAGE_KV;
  static constexpr int OFF_SX = OFF_SC + NSTAGE * SC_BYTES;
  static constexpr int OFF_PID = OFF_SX + SX_BYTES;
  static constexpr int OFF_BAR = OFF_PID + MAX_TPS * 4;
  static constexpr int SMEM = OFF_BAR + 2 * NSTAGE * 8;
  static constexpr int SMEM_ALLOC = SMEM + 1024;
  static_assert(NT >= 1 && NCW % NT == 0, "step shape");
  static_assert(QK_COLS % 32 == 0 && PV_COLS % 32 == 0, "warp column split");
};

struct DecK {
  const __nv_bfloat16* q;
  const int32_t* block_table;
  const int32_t* seq_lens;
  __nv_bfloat16* out;
  float* lse;
  float* o_part;
  float* ml_part;
  unsigned int* err;
  int B, Hq, Hkv, g, head_chunks, kind, window, page_size, tiles_per_page, num_pages;
  int max_pages_per_seq, max_seq_len, tiles_per_split, splits;
  float scale_log2;   // sm_scale * log2(e)
};

// Visible tile range [t_first, t_end) of a sequence of length L (already cut
// to the bound), and its first visible position lo.
__device__ __forceinline__ void seq_tiles(int L, int kind, int window, int& lo, int& t_first, int& t_end) {
  lo = (kind == FA_SLIDING) ? max(0, L - window) : 0;
  t_first = lo / kTile;
  t_end = (L - 1) / kTile + 1;
}

// int8 x4 (a 32-bit word) -> two fp16x2 words holding the exact integers.
// sel picks the bytes: 0x4140 -> (b0, b1), 0x4342 -> (b2, b3), 0x4240 -> (b0, b2), 0x4341 -> (b1, b3).
__device__ __forceinline__ uint32_t i8pair_to_f16x2(uint32_t biased, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(biased), "r"(0x64646464u), "r"(sel));
  // (0x64 << 8 | u) as fp16 is 1024 + u with u = c + 128; subtract 1152 to get c.
  __half2 h = *reinterpret_cast<__half2*>(&r);
  h = __hsub2(h, __half2(__float2half(1152.0f), __float2half(1152.0f)));
  return *reinterpret_cast<uint32_t*>(&h);
}

template <int D, int KV>
__global__ void __launch_bounds__(160, 2)
    decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_ks, const __grid_constant__ CUtensorMap tm_vs,
                  const DecK p) {
  using C = DecCfg<D, KV>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* sx = reinterpret_cast<float*>(smem + C::OFF_SX);
  int* pid = reinterpret_cast<int*>(smem + C::OFF_PID);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + C::NSTAGE;
  __shared__ int abort_flag;

  const int split = blockIdx.x;
  const int h = blockIdx.y / p.head_chunks, chunk = blockIdx.y % p.head_chunks;
  const int b = blockIdx.z;
  const int head0 = h * p.g + chunk * 8;
  const int nheads = min(8, p.g - chunk * 8);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;

  int L = __ldg(p.seq_lens + b);
  if (L > p.max_seq_len) {
    if (threadIdx.x == 0 && split == 0 && blockIdx.y == 0) atomicOr(p.err, FA_DEV_ERR_BOUND);
    L = p.max_seq_len;
  }
  const bool direct = (p.o_part == nullptr);   // one split: write the final output here
  if (L <= 0) {
    if (direct && split == 0) {
      for (int i = threadIdx.x; i < nheads * D; i += blockDim.x)
        p.out[(static_cast<size_t>(b) * p.Hq + head0 + i / D) * D + i % D] = __float2bfloat16(0.0f);
      if (p.lse && threadIdx.x < nheads) p.lse[static_cast<size_t>(b) * p.Hq + head0 + threadIdx.x] = -INFINITY;
    }
    return;
  }
  const int qpos = L - 1;
  int lo, t_first, t_end;
  seq_tiles(L, p.kind, p.window, lo, t_first, t_end);
  const int t0 = t_first + split * p.tiles_per_split;
  const int t1 = min(t0 + p.tiles_per_split, t_end);
  if (t0 >= t1) return;
  const int nsteps = (t1 - t0 + C::NT - 1) / C::NT;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NSTAGE; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C::NCW);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == C::NCW) {
    // ------------------------------------------------------------ producer
    const int32_t* bt = p.block_table + static_cast<size_t>(b) * p.max_pages_per_seq;
    bool bad = false;
    for (int k = lane; k < t1 - t0; k += 32) {
      int page = __ldg(bt + (t0 + k) / p.tiles_per_page);
      if (page < 0 || page >= p.num_pages) {
        bad = true;
        page = -1;   // the TMA box then lies outside the tensor and reads zeros
      }
      pid[k] = page;
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(p.err, FA_DEV_ERR_PAGE);
    __syncwarp();
    if (lane == 0) {
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      const uint64_t pol = l2_policy_evict_first();
      int issued = 0;
      for (int i = 0; i < nsteps; ++i) {
        const int st = i % C::NSTAGE;
        if (!mbar_wait(&empty[st], ((i / C::NSTAGE) & 1) ^ 1)) {
          atomicOr(p.err, FA_DEV_ERR_TIMEOUT);
          break;
        }
        const int ntl = min(C::NT, t1 - (t0 + i * C::NT));
        mbar_arrive_expect_tx(&full[st], ntl * (2 * C::TILE_BYTES + (KV ? 128 : 0)));
        uint8_t* kdst = smem + st * C::STAGE_KV;
        uint8_t* vdst = kdst + C::NT * C::TILE_BYTES;
        for (int t = 0; t < ntl; ++t) {
          const int tile = t0 + i * C::NT + t;
          const int row0 = (pid[tile - t0] * p.Hkv + h) * p.page_size + (tile % p.tiles_per_page) * kTile;
#pragma unroll
          for (int blk = 0; blk < C::NBLK; ++blk) {
            tma_load_3d(kdst + t * C::TILE_BYTES + blk * 2048, &tm_k, &full[st], 0, blk, row0, pol);
            tma_load_3d(vdst + t * C::TILE_BYTES + blk * 2048, &tm_v, &full[st], 0, blk, row0, pol);
          }
          if constexpr (KV) {
            float* sc = reinterpret_cast<float*>(smem + C::OFF_SC + st * C::SC_BYTES);
            tma_load_2d(sc + t * 32, &tm_ks, &full[st], 0, row0 / kTile, pol);
            tma_load_2d(sc + (C::NT + t) * 32, &tm_vs, &full[st], 0, row0 / kTile, pol);
          }
        }
        ++issued;
      }
      // drain: no bulk copy may still be landing when the CTA exits
      for (int i = max(0, issued - C::NSTAGE); i < issued; ++i)
        if (!mbar_wait(&full[i % C::NSTAGE], (i / C::NSTAGE) & 1)) atomicOr(p.err, FA_DEV_ERR_TIMEOUT);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int qk_tile = warp % C::NT;
  const int qk_d0 = (warp / C::NT) * C::QK_COLS;
  const int pv_d0 = warp * C::PV_COLS;

  // Q^T fragments (B operand), zero for padded heads.
  constexpr int QF = KV ? C::QK_COLS / 32 : C::QK_COLS / 16;
  uint32_t qf[QF][KV ? 4 : 2];
  {
    const bool hv = gid < nheads;
    const __nv_bfloat16* qrow = p.q + (static_cast<size_t>(b) * p.Hq + head0 + (hv ? gid : 0)) * D;
#pragma unroll
    for (int kk = 0; kk < QF; ++kk) {
      if constexpr (!KV) {
        const int d = qk_d0 + kk * 16 + 2 * tig;
        qf[kk][0] = hv ? __ldg(reinterpret_cast<const uint32_t*>(qrow + d)) : 0u;
        qf[kk][1] = hv ? __ldg(reinterpret_cast<const uint32_t*>(qrow + d + 8)) : 0u;
      } else {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int d = qk_d0 + kk * 32 + half * 16 + 4 * tig;
          uint2 w = hv ? __ldg(reinterpret_cast<const uint2*>(qrow + d)) : make_uint2(0u, 0u);
          qf[kk][2 * half + 0] = pack_f16x2(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u));
          qf[kk][2 * half + 1] = pack_f16x2(__uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
        }
      }
    }
  }

  float o[C::PV_MT][4];
#pragma unroll
  for (int i = 0; i < C::PV_MT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
  float m_run = -INFINITY, l_run = 0.0f, sigma = 1.0f;

  for (int i = 0; i < nsteps; ++i) {
    const int st = i % C::NSTAGE;
    const int buf = i & 1;
    const int tile0 = t0 + i * C::NT;
    const int ntl = min(C::NT, t1 - tile0);
    const uint8_t* ks = smem + st * C::STAGE_KV;
    const uint8_t* vs = ks + C::NT * C::TILE_BYTES;
    const float* scl = reinterpret_cast<const float*>(smem + C::OFF_SC + st * C::SC_BYTES);
    const bool ok = mbar_wait(&full[st], (i / C::NSTAGE) & 1);
    if (!ok && lane == 0) {
      abort_flag = 1;
      atomicOr(p.err, FA_DEV_ERR_TIMEOUT);
    }

    // ---- partial S^T over this warp's columns
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (ok && qk_tile < ntl) {
      const uint8_t* kt = ks + qk_tile * C::TILE_BYTES;
      const int r = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
      for (int kk = 0; kk < QF; ++kk) {
        uint32_t a0, a1, a2, a3;
        if constexpr (!KV) {
          const int dc = qk_d0 + kk * 16 + (lane >> 4) * 8;
          ldsm_x4(smem_u32(kt + (dc >> 6) * 2048 + sw128(r, (dc & 63) >> 3)), a0, a1, a2, a3);
          mma_bf16(acc, a0, a1, a2, a3, qf[kk][0], qf[kk][1]);
        } else {
          const int dc = qk_d0 + kk * 32 + (lane >> 4) * 16;
          ldsm_x4(smem_u32(kt + (dc >> 7) * 2048 + sw128(r, (dc & 127) >> 4)), a0, a1, a2, a3);
          const uint32_t x0 = a0 ^ 0x80808080u, x1 = a1 ^ 0x80808080u;
          const uint32_t x2 = a2 ^ 0x80808080u, x3 = a3 ^ 0x80808080u;
          mma_f16(acc, i8pair_to_f16x2(x0, 0x4140), i8pair_to_f16x2(x1, 0x4140), i8pair_to_f16x2(x0, 0x4342),
                  i8pair_to_f16x2(x1, 0x4342), qf[kk][0], qf[kk][1]);
          mma_f16(acc, i8pair_to_f16x2(x2, 0x4140), i8pair_to_f16x2(x3, 0x4140), i8pair_to_f16x2(x2, 0x4342),
                  i8pair_to_f16x2(x3, 0x4342), qf[kk][2], qf[kk][3]);
        }
      }
    }
    float* sxw = sx + (buf * C::NCW + warp) * kTile * C::SX_STRIDE;
    *reinterpret_cast<float2*>(sxw + gid * C::SX_STRIDE + 2 * tig) = make_float2(acc[0], acc[1]);
    *reinterpret_cast<float2*>(sxw + (gid + 8) * C::SX_STRIDE + 2 * tig) = make_float2(acc[2], acc[3]);
    named_bar_sync(1, C::NCW * 32);
    if (*reinterpret_cast<volatile int*>(&abort_flag)) break;

    // ---- scores for this lane's head (gid) and keys {2tig, 2tig+1, 2tig+8, 2tig+9} of each tile
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
        for (int w = t; w < C::NCW; w += C::NT)
          v += sx[((buf * C::NCW + w) * kTile + key) * C::SX_STRIDE + gid];
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
    float alpha = (m_run == -INFINITY) ? 0.0f : ex2(m_run - m_new);
    float psum = 0.0f;
    uint32_t pf[C::NT][2];
    float vmax = 1.0f;
    if constexpr (KV) {
      float vm = 0.0f;
#pragma unroll
      for (int t = 0; t < C::NT; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (valid[t][e]) vm = fmaxf(vm, scl[(C::NT + t) * 32 + 2 * tig + (e & 1) + (e >> 1) * 8]);
      vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, 1));
      vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, 2));
      vmax = vm > 0.0f ? vm : 1.0f;
    }
#pragma unroll
    for (int t = 0; t < C::NT; ++t) {
      float pe[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        pe[e] = ex2(s[t][e] - m_new);
        if constexpr (KV) psum += pe[e];
        if constexpr (KV) {
          const float vsc = scl[(C::NT + t) * 32 + 2 * tig + (e & 1) + (e >> 1) * 8];
          pe[e] = valid[t][e] ? pe[e] * __fdividef(vsc, vmax) : 0.0f;
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
      ofac = alpha * __fdividef(sigma, vmax);
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

    if constexpr (!KV) {
      // masked keys have p = 0, but their V rows may hold anything (NaN
      // included): zero this warp's columns of those rows before the MMA
      if (tile0 * kTile < lo || (tile0 + ntl) * kTile - 1 > qpos) {
        constexpr int UNITS = C::PV_COLS / 8;   // 16-byte units per row slice
        uint8_t* vw = const_cast<uint8_t*>(vs);
        for (int t = 0; t < ntl; ++t) {
          for (int idx = lane; idx < kTile * UNITS; idx += 32) {
            const int r = idx / UNITS, u = idx % UNITS;
            const int pos = (tile0 + t) * kTile + r;
            if (pos < lo || pos > qpos) {
              const int dc = pv_d0 + u * 8;
              *reinterpret_cast<uint4*>(vw + t * C::TILE_BYTES + (dc >> 6) * 2048 + sw128(r, (dc & 63) >> 3)) =
                  make_uint4(0u, 0u, 0u, 0u);
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
      if constexpr (!KV) {
        const int r = (lane & 7) + (lane >> 4) * 8;
#pragma unroll
        for (int mt = 0; mt < C::PV_MT; ++mt) {
          const int dc = pv_d0 + mt * 16 + ((lane >> 3) & 1) * 8;
          uint32_t a0, a1, a2, a3;
          ldsm_x4_t(smem_u32(vt + (dc >> 6) * 2048 + sw128(r, (dc & 63) >> 3)), a0, a1, a2, a3);
          mma_bf16(o[mt], a0, a1, a2, a3, pf[t][0], pf[t][1]);
        }
      } else {
        const int r = (lane & 7) + (lane >> 4) * 8;
#pragma unroll
        for (int gi = 0; gi < C::PV_MT / 2; ++gi) {
          const int dc = pv_d0 + gi * 32 + ((lane >> 3) & 1) * 16;
          uint32_t r0, r1, r2, r3;
          ldsm_x4_t(smem_u32(vt + (dc >> 7) * 2048 + sw128(r, (dc & 127) >> 4)), r0, r1, r2, r3);
          r0 ^= 0x80808080u;
          r1 ^= 0x80808080u;
          r2 ^= 0x80808080u;
          r3 ^= 0x80808080u;
          mma_f16(o[2 * gi], i8pair_to_f16x2(r0, 0x4240), i8pair_to_f16x2(r1, 0x4240), i8pair_to_f16x2(r2, 0x4240),
                  i8pair_to_f16x2(r3, 0x4240), pf[t][0], pf[t][1]);
          mma_f16(o[2 * gi + 1], i8pair_to_f16x2(r0, 0x4341), i8pair_to_f16x2(r1, 0x4341),
                  i8pair_to_f16x2(r2, 0x4341), i8pair_to_f16x2(r3, 0x4341), pf[t][0], pf[t][1]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }

  // -------------------------------------------------------------- epilogue
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
  const int hA = 2 * tig, hB = 2 * tig + 1;
  const float lA = __shfl_sync(0xffffffffu, l_run, 8 * tig);
  const float lB = __shfl_sync(0xffffffffu, l_run, 8 * tig + 4);
  const float mA = __shfl_sync(0xffffffffu, m_run, 8 * tig);
  const float mB = __shfl_sync(0xffffffffu, m_run, 8 * tig + 4);
  // output column d of C-fragment row (gid + 8 * half) of O^T tile mt
  auto out_d = [&](int mt, int half) -> int {
    if constexpr (!KV) return pv_d0 + mt * 16 + gid + 8 * half;
    else return pv_d0 + (mt >> 1) * 32 + 16 * half + 2 * gid + (mt & 1);
  };
  if (direct) {
    const float iA = (lA > 0.f) ? sigma / lA : 0.f, iB = (lB > 0.f) ? sigma / lB : 0.f;
#pragma unroll
    for (int mt = 0; mt < C::PV_MT; ++mt)
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int d = out_d(mt, half);
        if (hA < nheads)
          p.out[(static_cast<size_t>(b) * p.Hq + head0 + hA) * D + d] = __float2bfloat16_rn(o[mt][2 * half] * iA);
        if (hB < nheads)
          p.out[(static_cast<size_t>(b) * p.Hq + head0 + hB) * D + d] =
              __float2bfloat16_rn(o[mt][2 * half + 1] * iB);
      }
    if (p.lse && warp == 0 && tig == 0 && gid < nheads)
      p.lse[static_cast<size_t>(b) * p.Hq + head0 + gid] = (m_run + __log2f(l_run)) * 0.69314718055994531f;
  } else {
#pragma unroll
    for (int mt = 0; mt < C::PV_MT; ++mt)
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int d = out_d(mt, half);
        if (hA < nheads)
          p.o_part[((static_cast<size_t>(b) * p.Hq + head0 + hA) * p.splits + split) * D + d] = o[mt][2 * half] * sigma;
        if (hB < nheads)
          p.o_part[((static_cast<size_t>(b) * p.Hq + head0 + hB) * p.splits + split) * D + d] =
              o[mt][2 * half + 1] * sigma;
      }
    if (warp == 0 && tig == 0 && gid < nheads) {
      float2* ml = reinterpret_cast<float2*>(p.ml_part) + (static_cast<size_t>(b) * p.Hq + head0 + gid) * p.splits + split;
      *ml = make_float2(m_run, l_run);
    }
  }
  (void)mA;
  (void)mB;
}

// Merge the splits of one (sequence, query head): M = max m_s,
// l = sum l_s 2^(m_s - M), out = sum o_s 2^(m_s - M) / l.
template <int D>
__global__ void __launch_bounds__(D / 4) combine_kernel(const DecK p) {
  const int b = blockIdx.x / p.Hq, j = blockIdx.x % p.Hq;
  int L = __ldg(p.seq_lens + b);
  if (L > p.max_seq_len) L = p.max_seq_len;
  const int d = threadIdx.x * 4;
  __nv_bfloat16* orow = p.out + (static_cast<size_t>(b) * p.Hq + j) * D;
  if (L <= 0) {
    *reinterpret_cast<uint2*>(orow + d) = make_uint2(0u, 0u);
    if (p.lse && threadIdx.x == 0) p.lse[static_cast<size_t>(b) * p.Hq + j] = -INFINITY;
    return;
  }
  int lo, t_first, t_end;
  seq_tiles(L, p.kind, p.window, lo, t_first, t_end);
  const int ns = min(p.splits, (t_end - t_first + p.tiles_per_split - 1) / p.tiles_per_split);
  const size_t base = (static_cast<size_t>(b) * p.Hq + j) * p.splits;
  const float2* ml = reinterpret_cast<const float2*>(p.ml_part) + base;
  float M = -INFINITY;
  for (int s = 0; s < ns; ++s) M = fmaxf(M, ml[s].x);
  float lsum = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = 0; s < ns; ++s) {
    const float2 v = ml[s];
    const float w = ex2(v.x - M);
    lsum += v.y * w;
    const float4 x = *reinterpret_cast<const float4*>(p.o_part + (base + s) * D + d);
    acc.x += x.x * w;
    acc.y += x.y * w;
    acc.z += x.z * w;
    acc.w += x.w * w;
  }
  const float inv = lsum > 0.f ? 1.0f / lsum : 0.f;
  uint2 packed;
  packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
  packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
  *reinterpret_cast<uint2*>(orow + d) = packed;
  if (p.lse && threadIdx.x == 0) p.lse[static_cast<size_t>(b) * p.Hq + j] = (M + __log2f(lsum)) * 0.69314718055994531f;
}

template <int D, int KV>
static cudaError_t launch_decode_t(const DecodeArgs& a, const DecK& k, cudaStream_t s) {
  using C = DecCfg<D, KV>;
  static unsigned int done = 0;
  cudaError_t e0 = set_smem_once(reinterpret_cast<const void*>(decode_kernel<D, KV>), C::SMEM_ALLOC, &done);
  if (e0 != cudaSuccess) return e0;
  dim3 grid(a.plan.splits, a.Hkv * a.plan.head_chunks, a.B);
  decode_kernel<D, KV><<<grid, 160, C::SMEM_ALLOC, s>>>(*a.tm_k, *a.tm_v, *a.tm_ks, *a.tm_vs, k);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || k.o_part == nullptr) return e;
  combine_kernel<D><<<a.B * a.Hq, D / 4, 0, s>>>(k);
  return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
  DecK k{};
  k.q = static_cast<const __nv_bfloat16*>(a.q);
  k.block_table = a.block_table;
  k.seq_lens = a.seq_lens;
  k.out = static_cast<__nv_bfloat16*>(a.out);
  k.lse = a.lse;
  k.o_part = a.plan.splits > 1 ? a.o_part : nullptr;
  k.ml_part = a.plan.splits > 1 ? a.ml_part : nullptr;
  k.err = a.err;
  k.B = a.B;
  k.Hq = a.Hq;
  k.Hkv = a.Hkv;
  k.g = a.Hq / a.Hkv;
  k.head_chunks = a.plan.head_chunks;
  k.kind = a.kind;
  k.window = a.window;
  k.page_size = a.page_size;
  k.tiles_per_page = a.page_size / kTile;
  k.num_pages = a.num_pages;
  k.max_pages_per_seq = a.max_pages_per_seq;
  k.max_seq_len = a.max_seq_len;
  k.tiles_per_split = a.plan.tiles_per_split;
  k.splits = a.plan.splits;
  k.scale_log2 = a.sm_scale * 1.4426950408889634f;
  if (a.kv_dtype == FA_KV_INT8) {
    if (a.D == 256) return launch_decode_t<256, 1>(a, k, s);
    return launch_decode_t<512, 1>(a, k, s);
  }
  if (a.D == 256) return launch_decode_t<256, 0>(a, k, s);
  return launch_decode_t<512, 0>(a, k, s);
}

}  // namespace fa
