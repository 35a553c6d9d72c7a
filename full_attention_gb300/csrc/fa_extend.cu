// Chunked-prefill / extend attention on the 5th-generation tensor cores.
//
// Sequence b brings n_b new tokens at positions P_b .. P_b + n_b - 1 on top of
// a paged prefix of P_b tokens.  Token i attends to prefix keys (from the
// slab, through the block table) and to chunk keys P_b + j, j <= i (from
// k_ext / v_ext), under the layer's mask: causal, and for sliding layers
// q_pos - kv_pos < W ("FreeToken PR #898", description: the extend kernel takes
// the current chunk from k_extend / v_extend; "unsloth gemma4_flex_inference.py"
// history, "block mask per attention regime").
//
// One CTA owns 128 query rows of one (sequence, KV head): T = 128 / g tokens
// times the g query heads that share the KV head (GQA packed into the M
// dimension, so each K/V tile serves all g heads), and one 256-column slice of
// the output (head_dim 512 uses two CTAs, each recomputing S over the full
// head_dim; a 128 x 512 fp32 O would fill all of tensor memory).  Roles:
//   warp 0      TMA producer: Q once (4-D map, rows = (token, head)); per
//               64-key tile the K tile in 64-column chunks and the V tile of
//               this CTA's output slice, from slab pages or from k_ext / v_ext;
//   warp 1      MMA issuer: S_j = Q K_j^T (tcgen05.mma, M=128, N=64, fp32 in
//               TMEM, double buffered), then O += P_{j-1} V_{j-1} with P read
//               from tensor memory and V as an MN-major operand (N=256);
//   warps 2-5   softmax: one query row per thread; load S from TMEM, mask,
//               online softmax in the log2 domain, write P (bf16) back into the
//               S buffer; rescale O in TMEM only when the running max grows by
//               more than 2^8, so rescales are rare; final normalisation and
//               bf16 store.
// Every wait is bounded; tensor memory is always freed.
#include <cfloat>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {

template <int D>
struct ExtCfg {
  static constexpr int M = 128;                 // query rows per CTA
  static constexpr int NK = 64;                 // keys per tile
  static constexpr int DS = 256;                // output columns per CTA
  static constexpr int KB = D / 64;             // 64-column blocks of head_dim
  static constexpr int Q_BYTES = M * D * 2;     // [KB][128][64] bf16
  static constexpr int KCH_BYTES = NK * 64 * 2; // one K chunk: 64 keys x 64 columns
  static constexpr int KSTAGES = 4;
  static constexpr int V_BYTES = NK * DS * 2;   // [4 blocks][64 keys][64 columns]
  static constexpr int VSTAGES = 2;
  static constexpr int OFF_K = Q_BYTES;
  static constexpr int OFF_V = OFF_K + KSTAGES * KCH_BYTES;
  static constexpr int OFF_BAR = OFF_V + VSTAGES * V_BYTES;
  // barriers: q_full, k_full[4], k_empty[4], v_full[2], v_empty[2], s_full[2], p_full[2], o_bar[2]
  static constexpr int NBAR = 1 + 2 * KSTAGES + 2 * VSTAGES + 2 + 2 + 2;
  static constexpr int SMEM = OFF_BAR + NBAR * 8 + 16;
  static constexpr int SMEM_ALLOC = SMEM + 1024;
  static constexpr int NTHR = 6 * 32;
  // tensor memory columns: O [0, 256), S/P buffers [256, 320) and [320, 384)
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t S_COL0 = 256;
  static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
};

struct ExtK {
  const int32_t* qo_indptr;
  const int32_t* prefix_lens;
  const int32_t* block_table;
  __nv_bfloat16* out;
  float* lse;
  unsigned int* err;
  int B, Hq, Hkv, g, T, kind, window, page_size, tiles_per_page, num_pages, max_pages_per_seq;
  int max_q_len, max_prefix_len, dslices, early_metadata;
  float scale_log2;
};

// The key tiles one CTA walks: prefix tiles (16-aligned starts, from the
// slab) then chunk tiles (64-aligned relative to P, from k_ext / v_ext).
struct ExtPlan {
  int b, h, ds, t0, n, P, qo0;
  int kmin, kmax;          // visible key positions of the CTA's rows
  int a0, np;              // first prefix tile start, number of prefix tiles
  int c0, nc;              // first chunk tile start (absolute position), number of chunk tiles
  __device__ int tiles() const { return np + nc; }
  __device__ bool prefix(int j) const { return j < np; }
  __device__ int start(int j) const { return j < np ? a0 + 64 * j : c0 + 64 * (j - np); }
};

__device__ __forceinline__ bool ext_plan(const ExtK& p, ExtPlan& x) {
  x.b = blockIdx.z;
  x.h = blockIdx.y / p.dslices;
  x.ds = blockIdx.y % p.dslices;
  x.t0 = blockIdx.x * p.T;
  x.qo0 = __ldg(p.qo_indptr + x.b);
  x.n = __ldg(p.qo_indptr + x.b + 1) - x.qo0;
  x.P = __ldg(p.prefix_lens + x.b);
  bool bad = false;
  if (x.n > p.max_q_len) { x.n = p.max_q_len; bad = true; }
  if (x.P > p.max_prefix_len) { x.P = p.max_prefix_len; bad = true; }
  if (x.P < 0 || x.n < 0) { x.P = max(x.P, 0); x.n = max(x.n, 0); bad = true; }
  if (bad && threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) atomicOr(p.err, FA_DEV_ERR_BOUND);
  if (x.t0 >= x.n) return false;
  const int q_first = x.P + x.t0;
  const int q_last = x.P + min(x.t0 + p.T, x.n) - 1;
  x.kmin = (p.kind == FA_SLIDING) ? max(0, q_first - p.window + 1) : 0;
  x.kmax = q_last;
  x.np = 0;
  x.a0 = (x.kmin / 16) * 16;
  if (x.kmin < x.P) x.np = (x.P - x.a0 + 63) / 64;
  const int cfirst = max(x.kmin, x.P);
  x.c0 = x.P + ((cfirst - x.P) / 64) * 64;
  x.nc = (x.kmax >= x.c0) ? (x.kmax - x.c0) / 64 + 1 : 0;
  return true;
}

template <int D>
__global__ void __launch_bounds__(ExtCfg<D>::NTHR, 1)
    extend_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_kx,
                  const __grid_constant__ CUtensorMap tm_vx, const ExtK p) {
  using C = ExtCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* qs = smem;
  uint8_t* kring = smem + C::OFF_K;
  uint8_t* vring = smem + C::OFF_V;
  uint64_t* q_full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* k_full = q_full + 1;
  uint64_t* k_empty = k_full + C::KSTAGES;
  uint64_t* v_full = k_empty + C::KSTAGES;
  uint64_t* v_empty = v_full + C::VSTAGES;
  uint64_t* s_full = v_empty + C::VSTAGES;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_bar = p_full + 2;
  __shared__ uint32_t tmem_slot;
  __shared__ uint64_t done_bar;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (!p.early_metadata) griddep_wait();
  griddep_launch_dependents();
  ExtPlan x;
  if (!ext_plan(p, x)) return;
  const int nt = x.tiles();

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < C::KSTAGES; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < C::VSTAGES; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 4);
    }
    mbar_init(&o_bar[0], 1);
    mbar_init(&o_bar[1], 1);
    mbar_init(&done_bar, 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  griddep_wait();   // from here on q, k, v, the slab and the outputs are touched

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = l2_policy_evict_last();   // K/V tiles are shared by the CTAs of a (sequence, head)
    int kc = 0, vc = 0;
    bool ok = true;
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      mbar_arrive_expect_tx(q_full, C::Q_BYTES);
      for (int kb = 0; kb < C::KB; ++kb)
        tma_load_4d(qs + kb * (C::M * 128), &tm_q, q_full, 0, x.h * p.g, x.qo0 + x.t0, kb, pol);
    }
    const int32_t* bt = p.block_table + static_cast<size_t>(x.b) * p.max_pages_per_seq;
    for (int j = 0; ok && j < nt; ++j) {
      const int st0 = x.start(j);
      const bool pre = x.prefix(j);
      int pid = -1;
      if (pre && lane < 4) {
        const int pos = st0 + 16 * lane;
        if (pos < x.P) {
          pid = __ldg(bt + pos / p.page_size);
          if (pid < 0 || pid >= p.num_pages) {
            atomicOr(p.err, FA_DEV_ERR_PAGE);
            pid = -1;   // outside the tensor: the box reads zeros
          }
        }
      }
      int row0[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int pg = __shfl_sync(0xffffffffu, pid, i);
        row0[i] = (pg * p.Hkv + x.h) * p.page_size + ((st0 + 16 * i) % p.page_size);
      }
      const int xrow = x.qo0 + (st0 - x.P);   // chunk tiles: first token row in k_ext / v_ext
      if (lane == 0) {
        for (int kb = 0; ok && kb < C::KB; ++kb, ++kc) {
          const int st = kc % C::KSTAGES;
          ok = mbar_wait(&k_empty[st], ((kc / C::KSTAGES) & 1) ^ 1);
          if (!ok) break;
          mbar_arrive_expect_tx(&k_full[st], C::KCH_BYTES);
          uint8_t* dst = kring + st * C::KCH_BYTES;
          if (pre) {
#pragma unroll
            for (int i = 0; i < 4; ++i) tma_load_3d(dst + i * 2048, &tm_k, &k_full[st], 0, kb, row0[i], pol);
          } else {
            tma_load_4d(dst, &tm_kx, &k_full[st], 0, kb, x.h, xrow, pol);
          }
        }
        if (ok) {
          const int vs = vc % C::VSTAGES;
          ok = mbar_wait(&v_empty[vs], ((vc / C::VSTAGES) & 1) ^ 1);
          if (ok) {
            mbar_arrive_expect_tx(&v_full[vs], C::V_BYTES);
            uint8_t* dst = vring + vs * C::V_BYTES;
#pragma unroll
            for (int i4 = 0; i4 < 4; ++i4) {
              const int blk = x.ds * 4 + i4;
              if (pre) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                  tma_load_3d(dst + i4 * 8192 + i * 2048, &tm_v, &v_full[vs], 0, blk, row0[i], pol);
              } else {
                tma_load_4d(dst + i4 * 8192, &tm_vx, &v_full[vs], 0, blk, x.h, xrow, pol);
              }
            }
            ++vc;
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    if (lane == 0) {
      if (!ok) atomicOr(p.err, FA_DEV_ERR_TIMEOUT);
      // drain: no bulk copy may still be landing when the CTA exits
      if (!mbar_wait(q_full, 0)) atomicOr(p.err, FA_DEV_ERR_TIMEOUT);
      for (int i = max(0, kc - C::KSTAGES); i < kc; ++i)
        if (!mbar_wait(&k_full[i % C::KSTAGES], (i / C::KSTAGES) & 1)) atomicOr(p.err, FA_DEV_ERR_TIMEOUT);
      for (int i = max(0, vc - C::VSTAGES); i < vc; ++i)
        if (!mbar_wait(&v_full[i % C::VSTAGES], (i / C::VSTAGES) & 1)) atomicOr(p.err, FA_DEV_ERR_TIMEOUT);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idS = umma_idesc_bf16(C::M, C::NK, false);
      const uint32_t idO = umma_idesc_bf16(C::M, C::DS, true);
      bool ok = mbar_wait(q_full, 0);
      int kc = 0;
      auto pv = [&](int i) {
        const int sb = i & 1, vs = i % C::VSTAGES;
        ok = ok && mbar_wait(&p_full[sb], (i >> 1) & 1);
        ok = ok && mbar_wait(&v_full[vs], (i / C::VSTAGES) & 1);
        if (!ok) return;
        tc_fence_after();
        const uint32_t vbase = smem_u32(vring + vs * C::V_BYTES);
#pragma unroll
        for (int ks = 0; ks < C::NK / 16; ++ks)
          umma_ts(tmem, tmem + C::S_COL0 + sb * 64 + ks * 8, umma_desc_sw128(vbase + ks * 2048, 8192, 1024), idO,
                  (i > 0 || ks > 0) ? 1u : 0u);
        umma_commit(&v_empty[vs]);
        umma_commit(&o_bar[i & 1]);   // PV i completes phase i / 2 of o_bar[i & 1]
      };
      for (int j = 0; ok && j < nt; ++j) {
        const int sb = j & 1;
        if (j >= 2) ok = mbar_wait(&o_bar[j & 1], ((j - 2) >> 1) & 1);   // PV_{j-2} has read P from this buffer
        if (!ok) break;
        tc_fence_after();
        const uint32_t s_tmem = tmem + C::S_COL0 + sb * 64;
        for (int kb = 0; kb < C::KB; ++kb, ++kc) {
          const int st = kc % C::KSTAGES;
          ok = mbar_wait(&k_full[st], (kc / C::KSTAGES) & 1);
          if (!ok) break;
          tc_fence_after();
          const uint32_t qb = smem_u32(qs + kb * (C::M * 128));
          const uint32_t kbase = smem_u32(kring + st * C::KCH_BYTES);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            umma_ss(s_tmem, umma_desc_sw128(qb + ks * 32, 16, 1024), umma_desc_sw128(kbase + ks * 32, 16, 1024), idS,
                    (kb > 0 || ks > 0) ? 1u : 0u);
          umma_commit(&k_empty[st]);
        }
        if (!ok) break;
        umma_commit(&s_full[sb]);
        if (j >= 1) pv(j - 1);
      }
      if (ok && nt >= 1) pv(nt - 1);
      if (!ok) atomicOr(p.err, FA_DEV_ERR_TIMEOUT);
      // every MMA this thread issued has finished before tensor memory is freed
      umma_commit(&done_bar);
      if (!mbar_wait(&done_bar, 0)) atomicOr(p.err, FA_DEV_ERR_TIMEOUT);
    }
  } else {
    // ------------------------------------------------------------- softmax
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;   // query row = tensor-memory lane
    const int tl = r / p.g, hj = r % p.g;
    const int t = x.t0 + tl;
    const bool row_ok = t < x.n;
    const int qpos = x.P + t;
    const uint32_t trow = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      const int sb = j & 1;
      const uint32_t s_col = C::S_COL0 + sb * 64;
      ok = mbar_wait(&s_full[sb], (j >> 1) & 1);
      if (__any_sync(0xffffffffu, !ok)) break;
      tc_fence_after();
      uint32_t sr[2][32];
      tmem_ld32(trow + s_col, sr[0]);
      tmem_ld32(trow + s_col + 32, sr[1]);
      tmem_ld_wait();
      const int st0 = x.start(j);
      const bool pre = x.prefix(j);
      float sv[64];
      float mt = -INFINITY;
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const int kp = st0 + c;
        bool v = row_ok && kp <= qpos && (p.kind == FA_FULL || qpos - kp < p.window);
        if (pre) v = v && kp < x.P;
        sv[c] = v ? __uint_as_float(sr[c >> 5][c & 31]) * p.scale_log2 : -INFINITY;
        mt = fmaxf(mt, sv[c]);
      }
      const float m_new = fmaxf(m_run, mt);
      const bool need = m_new > m_run + 8.0f;   // rescale only when the max grows by more than 2^8
      if (__any_sync(0xffffffffu, need && m_run > -INFINITY) && j > 0) {
        ok = mbar_wait(&o_bar[(j - 1) & 1], ((j - 1) >> 1) & 1);   // PV_{j-1} has finished writing O
        if (__any_sync(0xffffffffu, !ok)) break;
        tc_fence_after();
        const float f = (need && m_run > -INFINITY) ? ex2(m_run - m_new) : 1.0f;
#pragma unroll 1
        for (int c = 0; c < C::DS; c += 32) {
          uint32_t o[32];
          tmem_ld32(trow + c, o);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
          tmem_st32(trow + c, o);
        }
        tmem_st_wait();
      }
      if (need) {
        l_run = (m_run > -INFINITY) ? l_run * ex2(m_run - m_new) : 0.f;
        m_run = m_new;
      }
      uint32_t pk[32];
      float psum = 0.f;
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float p0 = (m_run > -INFINITY) ? ex2(sv[2 * c] - m_run) : 0.f;
        const float p1 = (m_run > -INFINITY) ? ex2(sv[2 * c + 1] - m_run) : 0.f;
        pk[c] = pack_bf16x2(p0, p1);
        // the denominator sums the bf16-rounded weights the PV MMA uses
        psum += __uint_as_float(pk[c] << 16) + __uint_as_float(pk[c] & 0xffff0000u);
      }
      l_run += psum;
      tmem_st32(trow + s_col, pk);
      tmem_st_wait();
      if (pre && st0 + 64 > x.P && (x.P & 15) != 0) {
        // the slab rows of the last prefix page past P hold whatever the slots
        // held before; their P is 0, but zero them so no NaN enters the MMA
        // (each warp zeroes its share and fences before arriving on p_full,
        // which the MMA issuer waits for before reading V)
        const int vs = j % C::VSTAGES;
        ok = mbar_wait(&v_full[vs], (j / C::VSTAGES) & 1);
        if (__any_sync(0xffffffffu, !ok)) break;
        const int r0 = x.P - st0, r1 = min(64, ((x.P + 15) & ~15) - st0);
        uint8_t* vt = vring + vs * C::V_BYTES;
        const int units = (r1 - r0) * 4 * 8;   // rows x blocks x 16-byte units
        for (int e = threadIdx.x - 64; e < units; e += 128) {
          const int rr = r0 + e / 32, blk = (e / 8) % 4, u = e % 8;
          *reinterpret_cast<uint4*>(vt + blk * 8192 + sw128(rr, u)) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[sb]);
    }
    // ------------------------------------------------------------ epilogue
    if (ok && nt > 0) ok = mbar_wait(&o_bar[(nt - 1) & 1], ((nt - 1) >> 1) & 1);
    if (__any_sync(0xffffffffu, !ok)) {
      if (lane == 0) atomicOr(p.err, FA_DEV_ERR_TIMEOUT);
    } else {
      tc_fence_after();
      const float inv = (l_run > 0.f) ? 1.0f / l_run : 0.f;
      __nv_bfloat16* orow =
          p.out + (static_cast<size_t>(x.qo0 + t) * p.Hq + x.h * p.g + hj) * D + x.ds * C::DS;
#pragma unroll 1
      for (int c = 0; c < C::DS; c += 32) {
        uint32_t o[32];
        tmem_ld32(trow + c, o);
        tmem_ld_wait();
        if (row_ok) {
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            w[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            reinterpret_cast<uint4*>(orow + c)[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
        }
      }
      if (row_ok && x.ds == 0 && p.lse)
        p.lse[static_cast<size_t>(x.qo0 + t) * p.Hq + x.h * p.g + hj] =
            (m_run > -INFINITY && l_run > 0.f) ? (m_run + __log2f(l_run)) * 0.69314718055994531f : -INFINITY;
    }
  }

  // ------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D>
static cudaError_t launch_extend_t(const ExtendArgs& a, const ExtK& k, cudaStream_t s) {
  using C = ExtCfg<D>;
  static unsigned int done = 0;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(extend_kernel<D>), C::SMEM_ALLOC, &done);
  if (e != cudaSuccess) return e;
  const dim3 grid((a.max_q_len + k.T - 1) / k.T, a.Hkv * k.dslices, a.B);
  return launch_pdl(extend_kernel<D>, grid, dim3(C::NTHR), C::SMEM_ALLOC, s, a.tm_q, *a.tm_k, *a.tm_v, a.tm_kx,
                    a.tm_vx, k);
}

cudaError_t launch_extend(const ExtendArgs& a, cudaStream_t s) {
  ExtK k{};
  k.qo_indptr = a.qo_indptr;
  k.prefix_lens = a.prefix_lens;
  k.block_table = a.block_table;
  k.out = static_cast<__nv_bfloat16*>(a.out);
  k.lse = a.lse;
  k.err = a.err;
  k.B = a.B;
  k.Hq = a.Hq;
  k.Hkv = a.Hkv;
  k.g = a.Hq / a.Hkv;
  k.T = 128 / k.g;
  k.kind = a.kind;
  k.window = a.window;
  k.page_size = a.page_size;
  k.tiles_per_page = a.page_size / kTile;
  k.num_pages = a.num_pages;
  k.max_pages_per_seq = a.max_pages_per_seq;
  k.max_q_len = a.max_q_len;
  k.max_prefix_len = a.max_prefix_len;
  k.dslices = a.D / 256;
  k.early_metadata = a.early_metadata;
  k.scale_log2 = a.sm_scale * 1.4426950408889634f;
  if (a.D == 256) return launch_extend_t<256>(a, k, s);
  return launch_extend_t<512>(a, k, s);
}

}  // namespace fa
