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
// head_dim; a 128 x 512 fp32 O would fill all of tensor memory).
// Tensor memory (512 columns): O [0, 256), two S/P buffers [256, 384), and
// the first 256 columns of Q as bf16 pairs [384, 512), so S = Q K^T reads
// that part of Q from tensor memory and only the rest (head_dim 512) from
// shared memory; the freed shared memory deepens the K/V ring.  Roles:
//   warps 0-3   producers: Q once (4-D map, rows = (token, head)), its
//               shared-memory blocks in place and its tensor-memory blocks
//               into the ring's last slots for the softmax warps to move;
//               per 64-key tile the K tile in 64-column chunks and the V
//               tile of this CTA's output slice, from slab pages or from
//               k_ext / v_ext, slot e by warp e % 4;
//   warp 4      MMA issuer (the whole warp walks the schedule, one elected
//               lane issues): S_j = Q K_j^T (tcgen05.mma, M=128, N=64, fp32
//               in TMEM, double buffered), then O += P_{j-1} V_{j-1} with P
//               read from tensor memory and V as an MN-major operand;
//   warps 5-12  softmax: two warps per row quarter, each thread one query
//               row and half of each tile's 64 columns; first move the row's
//               leading 256 Q values from the staging slots into tensor
//               memory; per tile load S, mask, online softmax in the log2
//               domain, write P (bf16) back into the S buffer; rescale O in
//               TMEM only when the running max grows by more than 2^8, so
//               rescales are rare; final normalisation, the rows staged in the
//               idle ring and copied out by bulk copies.
// Jobs (a 128-row block, a KV head and column slice, a sequence) form a 1-D
// grid, the longest row blocks first; with a split workspace bound, the jobs
// of a last wave that would leave more than half of the SMs idle run as two
// CTAs each over the two halves of their key tiles, merged by the second to
// finish.
// 8-bit slabs (int8 or fp8 per-token-head codes): every MMA operand is f16.
// A loader warp copies each slot as soon as it is free: a prefix slot's raw
// codes by TMA into the slot's upper half, a chunk slot's bf16 rows by TMA
// as in the bf16 path.  The four producer warps then rewrite the slot in
// place as exact f16 values (int8: a byte permute and one subtraction per
// pair; e4m3: the hardware pair conversion; chunk rows: bf16 to f16), each
// taking one 16-row group; the softmax warps convert Q to f16 (its
// shared-memory blocks in place).  The per-key scales never touch the
// operands: producer warp 0 puts each tile's K scale (times the softmax
// scale) and V scale into a small ring beside the tiles; the softmax
// multiplies the fp32 scores by the K scale and folds the V scale into P.
// Its exponent base then tracks the largest score plus the largest log2 V
// scale of the tile half and sits 2^7 below it, so the weighted P stays
// below 2^15 whatever the scales.  A q or chunk value f16 cannot hold
// (magnitude 65520 or more) saturates to +-65504 and sets FA_DEV_ERR_RANGE;
// stored prefix rows have no such limit.
// Every wait is bounded; tensor memory is always freed.
#include <algorithm>
#include <cfloat>

#include <cuda_fp8.h>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {

template <int D, int KV = FA_KV_BF16>
struct ExtCfg {
  static constexpr int M = 128;                 // query rows per CTA
  static constexpr int NK = 64;                 // keys per tile
  // Output columns per CTA.  Tensor memory (512 columns) holds O (DS
  // columns), two 64-column S/P buffers and as many 64-column blocks of Q
  // (bf16 pairs, 32 columns each) as fit; the rest of Q stays in shared
  // memory.  head_dim 512 uses two CTAs per 128-row block (each recomputes S);
  // four CTAs with 128 columns each would hold all of Q in tensor memory but
  // doubles the S work again, which costs more than it saves.
  static constexpr int DS = 256;
  static constexpr int NVB = DS / 64;           // 64-column V blocks per tile
  static constexpr int KB = D / 64;             // 64-column blocks of head_dim
  static constexpr int NQT = (512 - DS - 128) / 32 < KB ? (512 - DS - 128) / 32 : KB;   // Q blocks in tensor memory
  static constexpr int NQS = KB - NQT;          // Q blocks held in shared memory
  static constexpr int Q_BYTES = NQS * M * 128; // [NQS][128][64] bf16
  static constexpr int CHUNK = NK * 64 * 2;     // 64 keys x 64 columns: a K chunk or a V block
  static constexpr int CPS = D == 256 ? 4 : 2;  // chunks (column blocks) per ring slot
  static constexpr int SLOT = CPS * CHUNK;      // one ring slot: CPS chunks side by side
  static constexpr int BAR_BYTES = 1024;
  // 8-bit slabs: a ring of per-tile key scales, SCL_R tiles deep; per tile
  // 64 K scales x softmax scale, 64 V scales, and per half of the keys the
  // largest log2 V scale
  static constexpr bool Q8 = KV != FA_KV_BF16;
  static constexpr int SCL_R = 8;
  static constexpr int SCL_TILE = 3 * 64 * 4;
  static constexpr int SCL_BYTES = Q8 ? SCL_R * SCL_TILE : 0;
  // 8-bit slabs: a prefix slot's raw codes (CPS x 64 rows x 64 codes) land
  // in the slot's upper half, in 128-byte lines of 128 codes
  static constexpr int CODE_OFF = SLOT / 2;
  static constexpr int NPW = 4;                 // producer warps
  // the rest of shared memory is a ring of slots; per tile KB K chunks and 4 V blocks pass through it
  static constexpr int NSLOT = (232448 - 1024 - Q_BYTES - BAR_BYTES - SCL_BYTES) / SLOT;
  static constexpr int OFF_RING = Q_BYTES;
  static constexpr int OFF_BAR = OFF_RING + NSLOT * SLOT;
  static constexpr int OFF_SCL = OFF_BAR + BAR_BYTES;
  static constexpr int SMEM = OFF_SCL + SCL_BYTES;
  static constexpr int SMEM_ALLOC = SMEM + 1024;
  // 16-row groups 0 .. TMA_GROUPS - 1 of a prefix tile come by TMA, the
  // others by the producer warp's cp.async copies (two copy paths in parallel)
  static constexpr int TMA_GROUPS = 2;
  static constexpr int W_MMA = NPW;             // the MMA warp; the softmax warps follow it
  static constexpr int NSMX = 8;                // softmax warps: two per tensor-memory lane quarter
  // 8-bit slabs: one more warp, the loader, issues every slot's TMA copies
  // (the producer warps convert what lands); an SM sub-partition then holds
  // 4 warps at most, so the register budget (128) is unchanged
  static constexpr int W_LOAD = NPW + 1 + NSMX;
  static constexpr int NTHR = (NPW + 1 + NSMX + (Q8 ? 1 : 0)) * 32;
  // tensor memory columns: O [0, DS), S/P buffers [DS, DS + 64) and
  // [DS + 64, DS + 128), Q blocks 0..NQT-1 [DS + 128, 512) (32 columns of
  // bf16 pairs each)
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t S_COL0 = DS;
  static constexpr uint32_t Q_COL0 = DS + 128;
  static_assert(Q_COL0 + NQT * 32 == TMEM_COLS, "tensor memory budget");
  static_assert(SMEM_ALLOC <= 232448, "shared memory budget");
  static_assert((1 + 3 * NSLOT + 2 + 2 + 2 + 1 + 1 + 1 + 2 * SCL_R + 2) * 8 <= BAR_BYTES, "barrier space");
  // Q's tensor-memory blocks arrive by TMA into the ring's last QST slots
  // (the boxes' 128-byte-swizzled layout, 16 KB per block) and the softmax
  // warps move them into tensor memory; the producers' first fill of those
  // slots waits until they have
  static constexpr int QST = NQT * (M * 128) / SLOT;
  static constexpr int QST_OFF = (NSLOT - QST) * SLOT;
  static_assert(NQT * (M * 128) % SLOT == 0 && QST >= 1 && QST < NSLOT, "Q staging slots");
  static_assert(NSLOT >= KB / CPS + NVB / CPS, "a ring must hold one tile");
  // a producer warp's consecutive slots lie NPW ring positions apart; its
  // parity wait on a slot's empty barrier is sound only while that is at most
  // one lap of the ring (else the barrier may be two phases behind and the
  // parity of an older phase passes the wait early)
  static_assert(NPW <= NSLOT, "producer stride within one ring lap");
  static_assert(KB % CPS == 0 && NVB % CPS == 0, "slots hold whole groups of column blocks");
};

struct ExtK {
  const __nv_bfloat16* q;
  const uint8_t* k_slab;   // [rows][D] bf16 (or 8-bit codes), rows = (page * Hkv + head) * page_size + offset
  const uint8_t* v_slab;
  const float* k_scale;    // 8-bit slabs: [rows] fp32 scales
  const float* v_scale;
  const uint8_t* k_ext;    // [num_tokens][Hkv][D] bf16
  const uint8_t* v_ext;
  const int32_t* qo_indptr;
  const int32_t* prefix_lens;
  const int32_t* seq_lens;   // keys_in_pages: every key (the new tokens' included) is read from the slab
  const int32_t* block_table;
  __nv_bfloat16* out;
  float* lse;
  unsigned int* err;
  int B, Hq, Hkv, g, T, kind, window, page_size, tiles_per_page, num_pages, max_pages_per_seq;
  int max_q_len, max_prefix_len, dslices, early_metadata, num_tokens, keys_in_pages;
  float scale_log2;
  // Jobs (128-row block, KV head and column slice, sequence) are numbered
  // row block fastest (last block first), gx row blocks and gy (head,
  // slice) pairs per sequence.  Jobs from split_from on run as two CTAs, each over half of the
  // job's key tiles; the second of the two to finish merges both (an arrival
  // counter per split job).  Their partials: ws_o [job][2][8 lane groups][32
  // float4 columns][32 lanes] fp32, ws_ml [job][2][128 rows] (base, rounded
  // sum, unrounded sum, 0), ws_cnt [job], zero between launches.
  int gx, gy, split_from;
  float4* ws_o;
  float4* ws_ml;
  int* ws_cnt;
};

// The key tiles one CTA walks: prefix tiles (16-aligned starts, from the
// slab) then chunk tiles (tile-aligned relative to P, from k_ext / v_ext).
// The CTAs of one (sequence, KV head) read the same prefix tiles; each walks
// them from a different starting tile (rot), so at any moment they read
// different lines and the L2 slices share the load.  The softmax does not
// depend on the order of the tiles.
struct ExtPlan {
  int nk;                  // keys per tile
  int bx, b, h, ds, t0, n, P, qo0;
  int Pk;                  // keys [0, Pk) come from the slab (P, or all keys when keys_in_pages)
  int kmin, kmax;          // visible key positions of the CTA's rows
  int a0, np;              // first prefix tile start, number of prefix tiles
  int c0, nc;              // first chunk tile start (absolute position), number of chunk tiles
  int rot;                 // walk prefix tiles from tile rot, wrapping
  int j0, nl;              // this CTA's tiles: [j0, j0 + nl) of the walk
  int ks, s, slot;         // the job's CTAs (1 or 2), this one's index, split-job index
  __device__ int tiles() const { return nl; }
  __device__ bool prefix(int j) const { return j + j0 < np; }
  __device__ int start(int j) const {
    j += j0;
    if (j < np) {
      int k = j + rot;
      if (k >= np) k -= np;
      return a0 + nk * k;
    }
    return c0 + nk * (j - np);
  }
};

template <int NK>
__device__ __forceinline__ bool ext_plan(const ExtK& p, ExtPlan& x) {
  x.nk = NK;
  const int cta = static_cast<int>(blockIdx.x);
  int job = cta;
  x.ks = 1;
  x.s = 0;
  x.slot = -1;
  if (cta >= p.split_from) {
    job = p.split_from + (cta - p.split_from) / 2;
    x.s = (cta - p.split_from) & 1;
    x.ks = 2;
    x.slot = job - p.split_from;
  }
  // row blocks in descending order: a later block of a chunk sees more keys
  // (causal), so the launch runs the longest jobs first and leaves the
  // shortest for the last wave
  x.bx = p.gx - 1 - job % p.gx;
  const int hy = (job / p.gx) % p.gy;
  x.b = job / (p.gx * p.gy);
  x.h = hy / p.dslices;
  x.ds = hy % p.dslices;
  x.t0 = x.bx * p.T;
  x.qo0 = __ldg(p.qo_indptr + x.b);
  x.n = __ldg(p.qo_indptr + x.b + 1) - x.qo0;
  bool bad = false;
  if (x.n > p.max_q_len) { x.n = p.max_q_len; bad = true; }
  if (x.n < 0) { x.n = 0; bad = true; }
  if (p.keys_in_pages) {
    // the n new tokens are the sequence's last n positions, already stored;
    // max_prefix_len bounds the sequence length
    int L = __ldg(p.seq_lens + x.b);
    if (L > p.max_prefix_len) { L = p.max_prefix_len; bad = true; }
    if (L < x.n) { x.n = max(L, 0); bad = true; }
    x.P = L - x.n;
    x.Pk = L;
  } else {
    x.P = __ldg(p.prefix_lens + x.b);
    if (x.P > p.max_prefix_len) { x.P = p.max_prefix_len; bad = true; }
    if (x.P < 0) { x.P = 0; bad = true; }
    x.Pk = x.P;
  }
  // one report per sequence, from its first job
  if (bad && threadIdx.x == 0 && job % (p.gx * p.gy) == 0 && x.s == 0) atomicOr(p.err, FA_DEV_ERR_BOUND);
  if (x.t0 >= x.n) return false;
  const int q_first = x.P + x.t0;
  const int q_last = x.P + min(x.t0 + p.T, x.n) - 1;
  x.kmin = (p.kind == FA_SLIDING) ? max(0, q_first - p.window + 1) : 0;
  x.kmax = q_last;
  x.np = 0;
  x.a0 = (x.kmin / 16) * 16;
  if (x.kmin < x.Pk) x.np = (x.Pk - x.a0 + NK - 1) / NK;
  const int cfirst = max(x.kmin, x.Pk);
  x.c0 = x.Pk + ((cfirst - x.Pk) / NK) * NK;
  x.nc = (x.kmax >= x.c0) ? (x.kmax - x.c0) / NK + 1 : 0;
  x.rot = x.np > 1 ? static_cast<int>((static_cast<unsigned>(x.bx) * 2u + x.ds) * 5u % static_cast<unsigned>(x.np)) : 0;
  // a split job's two CTAs take the first and second half of the walk; a
  // job of one tile runs whole on its first CTA
  const int nt = x.np + x.nc;
  if (x.ks > nt) x.ks = nt > 1 ? nt : 1;
  if (x.s >= x.ks) return false;
  x.j0 = x.s * nt / x.ks;
  x.nl = (x.s + 1) * nt / x.ks - x.j0;
  return true;
}

// 32 consecutive 8-bit codes (two 16-byte words) as exact f16 values, packed
// in pairs (lower column in the lower half).  int8: with u = c + 128 (the
// byte xor 0x80), the f16 bit pattern 0x6400 | u is 1024 + u, so one
// subtraction of 1152 per pair leaves c exactly; e4m3: the hardware pair
// conversion (every e4m3 value, subnormals included, is an f16 normal).
template <int KV>
__device__ __forceinline__ void codes32(const uint4 (&w)[2], uint32_t (&out)[16]) {
  const uint32_t word[8] = {w[0].x, w[0].y, w[0].z, w[0].w, w[1].x, w[1].y, w[1].z, w[1].w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if constexpr (KV == FA_KV_INT8) {
      const uint32_t u = word[i] ^ 0x80808080u;
      const __half2 off = __half2(__ushort_as_half(0x6480u), __ushort_as_half(0x6480u));   // 1152
      uint32_t lo, hi;
      asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(lo) : "r"(u), "r"(0x64646464u));
      asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(hi) : "r"(u), "r"(0x64646464u));
      const __half2 a = __hsub2(*reinterpret_cast<const __half2*>(&lo), off);
      const __half2 b = __hsub2(*reinterpret_cast<const __half2*>(&hi), off);
      out[2 * i] = *reinterpret_cast<const uint32_t*>(&a);
      out[2 * i + 1] = *reinterpret_cast<const uint32_t*>(&b);
    } else {
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(word[i] >> (16 * b)), __NV_E4M3);
        out[2 * i + b] = static_cast<uint32_t>(hr.x) | (static_cast<uint32_t>(hr.y) << 16);
      }
    }
  }
}

// 32 consecutive bf16 values (four 16-byte words) as f16 pairs (saturating);
// returns nonzero if any of them lies past the f16 range.
__device__ __forceinline__ uint32_t bf16_to_f16_32(const uint4 (&w)[4], uint32_t (&out)[16]) {
  const uint32_t word[16] = {w[0].x, w[0].y, w[0].z, w[0].w, w[1].x, w[1].y, w[1].z, w[1].w,
                             w[2].x, w[2].y, w[2].z, w[2].w, w[3].x, w[3].y, w[3].z, w[3].w};
  uint32_t big = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    big |= bf16x2_past_f16(word[i]);
    out[i] = pack_f16x2_sat(__uint_as_float(word[i] << 16), __uint_as_float(word[i] & 0xffff0000u));
  }
  return big;
}

// The two softmax warps of a row (each holding half of a tile's scores)
// must compute their weights against one common base at least the row's
// largest scaled score.  Each publishes its half's maximum rounded up to an
// integer (log2 units) as an int16, so the common base max(a, b) exceeds the
// true maximum by less than 1 and the largest weight stays in (0.5, 1] (a
// rounding to bf16 would leave up to |max| / 256 of excess, which makes f16
// weights underflow once scores reach a few thousand).  INT16_MIN stands for
// "no visible key"; a maximum past +-32767 saturates and is reported.
__device__ __forceinline__ short max_code(float m, bool& out_of_range) {
  if (m == -INFINITY) return static_cast<short>(-32768);
  const float c = ceilf(m);
  out_of_range |= !(c <= 32767.f && c >= -32767.f);
  return static_cast<short>(fminf(fmaxf(c, -32767.f), 32767.f));
}
__device__ __forceinline__ float max_decode(short c) { return c == -32768 ? -INFINITY : static_cast<float>(c); }

// One bulk copy from shared to global memory (both addresses 16-byte
// aligned, size a multiple of 16), tracked by this thread's bulk group.
__device__ __forceinline__ void bulk_store(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(reinterpret_cast<uint64_t>(dst)),
               "r"(smem_u32(src)), "r"(bytes)
               : "memory");
}
// Wait until every bulk copy this thread issued has read its shared-memory source.
__device__ __forceinline__ void bulk_store_drain() {
  asm volatile("cp.async.bulk.commit_group;\n\tcp.async.bulk.wait_group.read 0;" ::: "memory");
}

template <int D, int KV>
__global__ void __launch_bounds__(ExtCfg<D, KV>::NTHR, 1)
    extend_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_kx,
                  const __grid_constant__ CUtensorMap tm_vx, const ExtK p) {
  using C = ExtCfg<D, KV>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* qs = smem;
  uint8_t* ring = smem + C::OFF_RING;
  uint64_t* q_full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* full = q_full + 1;          // [NSLOT]
  uint64_t* empty = full + C::NSLOT;    // [NSLOT]
  uint64_t* s_full = empty + C::NSLOT;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_bar = p_full + 2;
  uint64_t* qt_full = o_bar + 2;        // the softmax warps have put Q into tensor memory
  uint64_t& done_bar = qt_full[1];      // every MMA has completed (before tensor memory is freed)
  uint32_t& tmem_slot = *reinterpret_cast<uint32_t*>(qt_full + 2);
  uint64_t* sc_full = qt_full + 3;      // 8-bit slabs: [SCL_R] a tile's scales are written
  uint64_t* sc_empty = sc_full + C::SCL_R;   // [SCL_R] the softmax has read them
  uint64_t* land = sc_empty + C::SCL_R;      // 8-bit slabs: [NSLOT] a slot's TMA data has landed
  uint64_t* qst_full = land + C::NSLOT;      // Q's tensor-memory blocks have landed in the staging slots
  uint64_t* q_free = qst_full + 1;           // the softmax warps have read them: the slots may be filled
  float* scl = reinterpret_cast<float*>(smem + C::OFF_SCL);   // [SCL_R][3][64]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (!p.early_metadata) griddep_wait();
  griddep_launch_dependents();
  ExtPlan x;
  if (!ext_plan<64>(p, x)) {
    // no work; the grid still ends only after the kernel before it (later
    // extend launches rely on that order for the split workspace)
    griddep_wait();
    return;
  }
  const int nt = x.tiles();
  // Producers: the first tile's page ids (block-table reads, index data the
  // dependency does not cover under early metadata, and already ordered after
  // it otherwise), issued before the set-up below so that the first K copies
  // can start as soon as the dependency resolves
  int pid0 = -1, off0 = 0;
  if ((warp < C::NPW || (C::Q8 && warp == C::W_LOAD)) && lane < 4 && nt > 0 && x.prefix(0)) {
    const int pos = x.start(0) + 16 * lane;   // a 16-row group lies in one page
    if (pos < x.Pk) {
      const int pg = pos / p.page_size;
      off0 = pos - pg * p.page_size;
      pid0 = ld_nc_early(p.block_table + static_cast<size_t>(x.b) * p.max_pages_per_seq + pg);
    }
  }

  if (warp == 0) {
    // the barriers, initialised by the lanes of warp 0 side by side: lane 0
    // the single ones, lane 1 + i ring slot i's, lane 16 + i scale slot i's
    static_assert(C::NSLOT <= 15 && C::SCL_R <= 16, "one lane per ring and scale slot");
    if (lane == 0) {
      mbar_init(q_full, 1);
      for (int i = 0; i < 2; ++i) {
        mbar_init(&s_full[i], 1);
        mbar_init(&p_full[i], C::NSMX);
      }
      mbar_init(&o_bar[0], 1);
      mbar_init(&o_bar[1], 1);
      mbar_init(qt_full, C::NSMX);
      mbar_init(&done_bar, 1);
      mbar_init(qst_full, 1);
      mbar_init(q_free, C::NSMX);
    } else if (lane <= C::NSLOT) {
      const int i = lane - 1;
      // bf16: the filling warp's lane 0 expect_tx + 32 lane arrivals; 8-bit:
      // one arrival per converting warp
      mbar_init(&full[i], C::Q8 ? C::NPW : 33);
      mbar_init(&empty[i], 1);
      if constexpr (C::Q8) mbar_init(&land[i], 32);   // the loader warp's 32 lanes
    } else if (C::Q8 && lane >= 16 && lane < 16 + C::SCL_R) {
      mbar_init(&sc_full[lane - 16], 32);        // the 32 lanes of producer warp 0
      mbar_init(&sc_empty[lane - 16], C::NSMX);  // one arrival per softmax warp
    }
    fence_mbar_init();
  }
  if (warp == C::W_MMA) tmem_alloc(&tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  griddep_wait();   // from here on q, k, v, the slab and the outputs are touched

  if (warp < C::NPW || (C::Q8 && warp == C::W_LOAD)) {
    // ----------------------------------------------------------- producers
    // Emission order = the MMA issuer's consumption order: K_0, then for each
    // t >= 1: K_t (if any) and V_{t-1}.  A slot is one 64-key x 64-column
    // block in the 128-byte-swizzled K-major layout, filled by one producer
    // warp (slot e by warp e % NPW): TMA boxes of 16 rows from the slab (one
    // per page), or one box of 64 rows from k_ext / v_ext.  A single thread
    // issues TMA copies at a rate that caps the fill far below what the MMAs
    // consume; four issuing warps do not.  The page that holds the prefix end
    // also holds slots past it (stale values, possibly NaN, that the PV MMA
    // would multiply by zero): its 16 rows are copied by the warp's lanes
    // with cp.async, zero-filling rows at or past the prefix end.
    // full[] counts 33 arrivals: lane 0's expect_tx, then 32 lane arrivals
    // (when their cp.async copies land, or at once when there are none).
    const int pw = warp < C::NPW ? warp : C::NPW;   // NPW: the 8-bit loader warp
    const uint64_t pol = l2_policy_evict_last();   // K/V rows are shared by the CTAs of a (sequence, head)
    if (threadIdx.x == 0) {
      // Q (bf16, both formats): its tensor-memory blocks into the staging
      // slots, the rest into its shared-memory blocks (8-bit slabs: the
      // softmax warps then rewrite those in place as f16)
      prefetch_tmap(&tm_q);
      mbar_arrive_expect_tx(qst_full, C::NQT * (C::M * 128));
      for (int kb = 0; kb < C::NQT; ++kb)
        tma_load_4d(ring + C::QST_OFF + kb * (C::M * 128), &tm_q, qst_full, 0, x.h * p.g, x.qo0 + x.t0, kb, pol);
      mbar_arrive_expect_tx(q_full, C::Q_BYTES);
      for (int kb = C::NQT; kb < C::KB; ++kb)
        tma_load_4d(qs + (kb - C::NQT) * (C::M * 128), &tm_q, q_full, 0, x.h * p.g, x.qo0 + x.t0, kb, pol);
    }
    if (lane == 0) {
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      prefetch_tmap(&tm_kx);
      prefetch_tmap(&tm_vx);
    }
    const int32_t* bt = p.block_table + static_cast<size_t>(x.b) * p.max_pages_per_seq;
    // Page of row group `lane` (lanes 0-3) of tile j and the group's offset in
    // it (pid -1: not a prefix row).  Looked up a tile ahead; the id is
    // checked where it is used.  Every producer warp resolves every tile, so
    // this per-tile work is kept short: one division per lane, done here,
    // and the lanes of a tile's four groups work in parallel.
    struct PageRef {
      int pid, off;
    };
    auto load_pid = [&](int j) -> PageRef {
      PageRef r{-1, 0};
      if (j < nt && x.prefix(j) && lane < 4) {
        const int pos = x.start(j) + 16 * lane;   // a 16-row group lies in one page
        if (pos < x.Pk) {
          const int q = pos / p.page_size;
          r.off = pos - q * p.page_size;
          r.pid = ld_nc_early(bt + q);
        }
      }
      return r;
    };
    struct TileSrc {
      int row0[4];   // slab row of each 16-row group (prefix tiles), -1: no page
      int lim;       // rows [0, lim) of the tile hold keys (prefix: < P)
      int wlim;      // rows below wlim precede every visible key of the CTA (window start): read as zero
      int bgroup;    // the group holding the prefix end inside it, -1: none
      bool prefix;
      int tok0;      // chunk tiles: first token row in k_ext / v_ext
    };
    auto tile_src = [&](int j, PageRef pr) {
      TileSrc ts;
      const int st0 = x.start(j);
      ts.prefix = x.prefix(j);
      ts.lim = ts.prefix ? x.Pk - st0 : x.n - (st0 - x.P);
      ts.bgroup = (ts.prefix && ts.lim < 64 && (ts.lim & 15) != 0) ? (ts.lim >> 4) : -1;
      ts.tok0 = x.qo0 + st0 - x.P;
      ts.wlim = ts.prefix ? max(0, x.kmin - st0) : 0;
      // lane g < 4 resolves group g's slab row; a bad page id reads as zeros
      int r0 = -1;
      if (lane < 4 && ts.prefix && 16 * lane < ts.lim) {
        if (pr.pid < 0 || pr.pid >= p.num_pages) {
          if (pw == 0) atomicOr(p.err, FA_DEV_ERR_PAGE);
        } else {
          r0 = (pr.pid * p.Hkv + x.h) * p.page_size + pr.off;
        }
      }
#pragma unroll
      for (int g = 0; g < 4; ++g) ts.row0[g] = __shfl_sync(0xffffffffu, r0, g);
      return ts;
    };
    // group g of a prefix tile goes by TMA: a whole page group of readable keys
    auto by_tma = [&](const TileSrc& ts, int g) {
      return g < C::TMA_GROUPS && g != ts.bgroup && ts.row0[g] >= 0 && 16 * g < ts.lim && 16 * g >= ts.wlim;
    };
    int e = 0;
    bool ok = true;
    // 8-bit slabs: convert slot e (its data has landed) in place and mark it
    // full.  The four producer warps share every slot: warp pw takes row
    // group pw (rows 16 pw .. 16 pw + 15), lane (row rr, half cpart) 32
    // columns of its row per column block h.  Prefix codes of block h sit in
    // the 128-byte lines of the slot's upper half (128 codes = blocks 2k2,
    // 2k2 + 1 per line, 16-byte pieces 128-byte swizzled); block h's f16 rows
    // are written over [h x 8 KB, (h + 1) x 8 KB), which covers code lines of
    // the same rows: the warp reads all its codes, syncs, then writes.  Rows
    // that hold no visible key become zero.  Chunk rows (bf16) convert piece
    // by piece in place; rows past the chunk become zero.
    auto convert = [&](const TileSrc& q) {
      const int sl = e % C::NSLOT;
      ok = __all_sync(0xffffffffu, mbar_wait(&land[sl], (e / C::NSLOT) & 1)) && ok;
      if (!ok) return;
      uint8_t* dst = ring + sl * C::SLOT;
      const int rr = lane >> 1, cpart = lane & 1;
      const int r = 16 * pw + rr;   // this warp's row group: pw
      if (q.prefix) {
        const int row0 = pw == 0 ? q.row0[0] : pw == 1 ? q.row0[1] : pw == 2 ? q.row0[2] : q.row0[3];
        const bool v = row0 >= 0 && r < q.lim && r >= q.wlim;
        // every code this lane converts is read before any write (the writes
        // of the last blocks cover the lines the codes sit in)
        uint4 w[C::CPS][2];
#pragma unroll
        for (int h = 0; h < C::CPS; ++h) {
          const uint8_t* cb = dst + C::CODE_OFF + (h >> 1) * 8192;
          const int c0 = (h & 1) * 4 + 2 * cpart;
          w[h][0] = v ? *reinterpret_cast<const uint4*>(cb + sw128(r, c0)) : make_uint4(0u, 0u, 0u, 0u);
          w[h][1] = v ? *reinterpret_cast<const uint4*>(cb + sw128(r, c0 + 1)) : make_uint4(0u, 0u, 0u, 0u);
        }
        __syncwarp();
#pragma unroll
        for (int h = 0; h < C::CPS; ++h) {
          uint32_t pk[16];
          codes32<KV>(w[h], pk);
#pragma unroll
          for (int u = 0; u < 4; ++u)
            *reinterpret_cast<uint4*>(dst + h * C::CHUNK + sw128(r, cpart * 4 + u)) =
                make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        }
      } else {
        uint32_t big = 0;
        const bool v = r < q.lim;
#pragma unroll
        for (int h = 0; h < C::CPS; ++h) {
          uint8_t* row = dst + h * C::CHUNK;
          uint4 w[4];
#pragma unroll
          for (int u = 0; u < 4; ++u)
            w[u] = v ? *reinterpret_cast<const uint4*>(row + sw128(r, cpart * 4 + u)) : make_uint4(0u, 0u, 0u, 0u);
          uint32_t pk[16];
          big |= bf16_to_f16_32(w, pk);
#pragma unroll
          for (int u = 0; u < 4; ++u)
            *reinterpret_cast<uint4*>(row + sw128(r, cpart * 4 + u)) =
                make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        }
        if (__any_sync(0xffffffffu, big != 0) && lane == 0) atomicOr(p.err, FA_DEV_ERR_RANGE);
      }
      // the generic writes, ordered for the MMA's async-proxy reads; full[]
      // counts one arrival per converting warp
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[sl]);
    };
    // one slot: column blocks blk0 .. blk0 + CPS - 1 (8 KB each)
    auto emit = [&](const TileSrc& ts, int blk0, bool is_v) {
      if constexpr (C::Q8) {
        // the loader copies every slot once it is empty (so copies run as far
        // ahead as the ring allows); the producer warps convert it together
        const int sl = e % C::NSLOT;
        if (pw == C::NPW) {
          bool w = true;
          if (lane == 0) {
            w = mbar_wait(&empty[sl], ((e / C::NSLOT) & 1) ^ 1);
            if (e < C::NSLOT && e >= C::NSLOT - C::QST) w = mbar_wait(q_free, 0) && w;   // Q's staging slots
          }
          ok = __shfl_sync(0xffffffffu, w, 0) && ok;
          if (ok) {
            uint8_t* dst = ring + sl * C::SLOT;
            if (ts.prefix) {
              // raw codes in the slot's upper half: TMA boxes of 16 rows x
              // 128 codes (128-byte swizzled), issued by lanes 0-3, one row
              // group each, for the groups that hold a readable key (the
              // conversion zeroes the other rows).  land[] counts lane 0's
              // expect_tx and 31 plain arrivals, then the bytes
              if (lane == 0) {
                int tx = 0;
#pragma unroll
                for (int g = 0; g < 4; ++g)
                  if (ts.row0[g] >= 0 && 16 * g < ts.lim && 16 * g + 16 > ts.wlim) tx += (C::CPS / 2) * 2048;
                mbar_arrive_expect_tx(&land[sl], tx);
              } else {
                mbar_arrive(&land[sl]);
              }
              __syncwarp();
              if (lane < 4) {
                const int g = lane;
                const int rg = g == 0 ? ts.row0[0] : g == 1 ? ts.row0[1] : g == 2 ? ts.row0[2] : ts.row0[3];
                if (rg >= 0 && 16 * g < ts.lim && 16 * g + 16 > ts.wlim)
#pragma unroll
                  for (int k2 = 0; k2 < C::CPS / 2; ++k2)
                    tma_load_3d(dst + C::CODE_OFF + k2 * 8192 + g * 2048, is_v ? &tm_v : &tm_k, &land[sl], 0,
                                blk0 / 2 + k2, rg, pol);
              }
            } else {
              // chunk rows (bf16), as in the bf16 path: lane 0's expect_tx
              // and 31 plain arrivals
              if (lane == 0) {
                mbar_arrive_expect_tx(&land[sl], C::SLOT);
                for (int h = 0; h < C::CPS; ++h)
                  tma_load_4d(dst + h * C::CHUNK, is_v ? &tm_vx : &tm_kx, &land[sl], 0, blk0 + h, x.h, ts.tok0, pol);
              } else {
                mbar_arrive(&land[sl]);
              }
            }
          }
          __syncwarp();
        } else if (ok) {
          convert(ts);
        }
        ++e;
        return;
      }
      if (e % C::NPW == pw) {
        const int sl = e % C::NSLOT;
        bool w = true;
        if (lane == 0) {
          w = mbar_wait(&empty[sl], ((e / C::NSLOT) & 1) ^ 1);
          if (e < C::NSLOT && e >= C::NSLOT - C::QST) w = mbar_wait(q_free, 0) && w;   // Q's staging slots
        }
        ok = __shfl_sync(0xffffffffu, w, 0) && ok;
        if (ok) {
          uint8_t* dst = ring + sl * C::SLOT;
          if (ts.prefix) {
            if (lane == 0) {
              int tx = 0;
#pragma unroll
              for (int g = 0; g < 4; ++g)
                if (by_tma(ts, g)) tx += C::CPS * 2048;
              mbar_arrive_expect_tx(&full[sl], tx);
#pragma unroll
              for (int h = 0; h < C::CPS; ++h)
#pragma unroll
                for (int g = 0; g < 4; ++g)
                  if (by_tma(ts, g))
                    tma_load_3d(dst + h * C::CHUNK + g * 2048, is_v ? &tm_v : &tm_k, &full[sl], 0, blk0 + h,
                                ts.row0[g], pol);
            }
            // groups without a page, past the prefix or before the window start
            // must read as zero: the slot holds older data, and the slab rows
            // there may hold anything (NaN included) that the PV MMA would
            // multiply by a zero weight
            const uint8_t* base = is_v ? p.v_slab : p.k_slab;
            bool any_cp = false;
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              if (by_tma(ts, g)) continue;
              any_cp = true;
              // 16 rows x 8 units per block: lane copies rows lane / 8 + 4 i, unit lane % 8
#pragma unroll
              for (int h = 0; h < C::CPS; ++h)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const int rr = (lane >> 3) + 4 * i, r = 16 * g + rr;
                  const bool v = ts.row0[g] >= 0 && r < ts.lim && r >= ts.wlim;
                  const uint8_t* src =
                      base + (v ? (static_cast<size_t>(ts.row0[g] + rr) * D + (blk0 + h) * 64) * 2 + (lane & 7) * 16 : 0);
                  cp_async16_zfill(dst + h * C::CHUNK + sw128(r, lane & 7), src, v, pol);
                }
            }
            if (any_cp) cp_async_mbar_arrive(&full[sl]);
            else if (lane == 0) mbar_arrive_n(&full[sl], 32);
          } else {
            if (lane == 0) {
              mbar_arrive_expect_tx(&full[sl], C::SLOT);
              for (int h = 0; h < C::CPS; ++h)
                tma_load_4d(dst + h * C::CHUNK, is_v ? &tm_vx : &tm_kx, &full[sl], 0, blk0 + h, x.h, ts.tok0, pol);
              mbar_arrive_n(&full[sl], 32);
            }
          }
        }
      }
      ++e;
    };
    // 8-bit slabs: warp 0 writes tile t's 64 key scales into scale slot
    // t % SCL_R once the softmax has released that slot's previous tile: lane
    // l handles keys l and l + 32.  ck = K scale x softmax scale (log2
    // domain), cv = V scale; a chunk key (bf16, as is) has ck = softmax scale
    // and cv = 1, a key that holds nothing visible ck = cv = 0.  Only warp 0
    // writes, tile by tile, so its parity wait on a slot's empty barrier is
    // never more than one lap behind; it never waits on anything that needs
    // the softmax of tile t or later before writing tile t's scales; and
    // before it waits for the softmax of tile t - SCL_R it converts every
    // slot it still holds, so that softmax never waits on this warp.
    float sk0 = 0.f, sk1 = 0.f, sv0 = 0.f, sv1 = 0.f;   // keys lane and lane + 32
    // key r of the tile lies in row group r / 16, whose slab row is row0
    auto scale_pair = [&](const TileSrc& ts, int r, int row0, float& k, float& v) {
      k = v = 0.f;
      if (ts.prefix) {
        if (row0 >= 0 && r < ts.lim && r >= ts.wlim) {
          const int row = row0 + (r & 15);
          k = __ldg(p.k_scale + row) * p.scale_log2;
          v = __ldg(p.v_scale + row);
        }
      } else if (r < ts.lim) {
        k = p.scale_log2;
        v = 1.0f;
      }
    };
    auto write_scales = [&](int t) {
      const int s = t % C::SCL_R;
      const uint32_t par = ((t / C::SCL_R) & 1) ^ 1;
      bool w = mbar_wait(&sc_empty[s], par);
      ok = __all_sync(0xffffffffu, w) && ok;
      if (!ok) return;
      float* dst = scl + s * (C::SCL_TILE / 4);
      dst[lane] = sk0;
      dst[lane + 32] = sk1;
      dst[64 + lane] = sv0;
      dst[96 + lane] = sv1;
      // the largest log2 V scale of each half's 32 keys: it only places the
      // exponent base, held at -90 or more so that the weights of keys with
      // tiny V scales (2^(score - base) < 2^105) and their sums stay finite
      float l0 = sv0 > 0.f ? fmaxf(__log2f(sv0), -90.f) : -INFINITY;
      float l1 = sv1 > 0.f ? fmaxf(__log2f(sv1), -90.f) : -INFINITY;
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        l0 = fmaxf(l0, __shfl_xor_sync(0xffffffffu, l0, o));
        l1 = fmaxf(l1, __shfl_xor_sync(0xffffffffu, l1, o));
      }
      if (lane < 2) dst[128 + lane] = lane == 0 ? l0 : l1;
      mbar_arrive(&sc_full[s]);
    };
    PageRef pid_next{pid0, off0};   // load_pid(0), read above
    TileSrc src_cur{}, src_prev{};
    for (int t = 0; ok && t <= nt; ++t) {
      if (t < nt) {
        const PageRef pid = pid_next;
        pid_next = load_pid(t + 1);   // a tile ahead
        src_cur = tile_src(t, pid);
        if constexpr (C::Q8)
          if (pw == 0) {
            const bool hi = lane >= 16;
            scale_pair(src_cur, lane, hi ? src_cur.row0[1] : src_cur.row0[0], sk0, sv0);
            scale_pair(src_cur, lane + 32, hi ? src_cur.row0[3] : src_cur.row0[2], sk1, sv1);
          }
        for (int kb = 0; ok && kb < C::KB; kb += C::CPS) emit(src_cur, kb, false);
        if constexpr (C::Q8)
          if (pw == 0 && ok) write_scales(t);
      }
      if (t >= 1)
        for (int i4 = 0; ok && i4 < C::NVB; i4 += C::CPS) emit(src_prev, x.ds * C::NVB + i4, true);
      src_prev = src_cur;
    }
    if (!ok && lane == 0) atomicOr(p.err, FA_DEV_ERR_TIMEOUT);
    // drain: no copy may still be landing when the CTA exits (8-bit slabs:
    // the loader waits for its copies, the converting warps issued none)
    asm volatile("cp.async.wait_all;" ::: "memory");
    if (lane == 0 && (!C::Q8 || pw == C::NPW)) {
      for (int i = max(0, e - C::NSLOT); i < e; ++i)
        if ((C::Q8 || i % C::NPW == pw) &&
            !mbar_wait(C::Q8 ? &land[i % C::NSLOT] : &full[i % C::NSLOT], (i / C::NSLOT) & 1))
          atomicOr(p.err, FA_DEV_ERR_TIMEOUT);
    }
    if (threadIdx.x == 0 && !(mbar_wait(q_full, 0) && mbar_wait(qst_full, 0))) atomicOr(p.err, FA_DEV_ERR_TIMEOUT);
  } else if (warp == C::W_MMA) {
    // ---------------------------------------------------------- MMA issuer
    // The whole warp walks the schedule and waits on the barriers, so slot
    // addresses and descriptors are warp-uniform; one elected lane (always
    // the same one) issues the MMAs and the commits that track them.
    // 8-bit slabs: Q, K, P and V are all f16 (dequantised values keep 11
    // significant bits); bf16 slabs: all bf16, as stored
    const uint32_t idS = KV == FA_KV_BF16 ? umma_idesc_bf16(C::M, C::NK, false) : umma_idesc_f16(C::M, C::NK, false);
    // the V blocks of a slot, LBO = CHUNK; P and V are f16 for 8-bit slabs
    const uint32_t idO = KV == FA_KV_BF16 ? umma_idesc_bf16(C::M, 64 * C::CPS, true)
                                          : umma_idesc_f16(C::M, 64 * C::CPS, true);
    bool ok = __all_sync(0xffffffffu, mbar_wait(q_full, 0) && mbar_wait(qt_full, 0));
    tc_fence_after();
    const uint64_t qd0 = umma_desc_sw128(smem_u32(qs), 16, 1024);   // Q's shared-memory blocks
    int e = 0;
    auto take = [&]() -> uint32_t {   // wait for the next ring slot, return its address
      const int sl = e % C::NSLOT;
      ok = __all_sync(0xffffffffu, ok && mbar_wait(&full[sl], (e / C::NSLOT) & 1));
      fence_proxy_async_smem();   // the cp.async writes, seen through the barrier, for the MMA's reads
      tc_fence_after();
      return smem_u32(ring + sl * C::SLOT);
    };
    auto give = [&]() {   // release the slot once the MMAs reading it complete
      if (elect_one()) umma_commit(&empty[e % C::NSLOT]);
      __syncwarp();
      ++e;
    };
    for (int t = 0; ok && t <= nt; ++t) {
      if (t < nt) {
        const int sb = t & 1;
        if (t >= 2) ok = __all_sync(0xffffffffu, mbar_wait(&o_bar[t & 1], ((t - 2) >> 1) & 1));   // PV_{t-2} has read P
        tc_fence_after();
        const uint32_t s_tmem = tmem + C::S_COL0 + sb * 64;
        for (int kp = 0; ok && kp < C::KB; kp += C::CPS) {
          const uint32_t sbase = take();   // K chunks kp .. kp + CPS - 1
          if (!ok) break;
          // one descriptor per slot; within it an operand at byte offset off
          // has descriptor d0 + off / 16 (start-address field, no carry: every
          // shared-memory address is below 256 KB)
          const uint64_t kd0 = umma_desc_sw128(sbase, 16, 1024);
          if (elect_one()) {
#pragma unroll
            for (int h = 0; h < C::CPS; ++h) {
              const int kb = kp + h;
              const uint64_t kd = kd0 + static_cast<uint64_t>(h * C::CHUNK / 16);
              if (kb < C::NQT) {   // A = Q block from tensor memory
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                  umma_ts(s_tmem, tmem + C::Q_COL0 + kb * 32 + ks * 8, kd + 2 * ks, idS, (kb > 0 || ks > 0) ? 1u : 0u);
              } else {             // A = Q block from shared memory
                const uint64_t qd = qd0 + static_cast<uint64_t>((kb - C::NQT) * (C::M * 128) / 16);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) umma_ss(s_tmem, qd + 2 * ks, kd + 2 * ks, idS, 1u);
              }
            }
          }
          __syncwarp();
          give();
        }
        if (!ok) break;
        if (elect_one()) umma_commit(&s_full[sb]);
        __syncwarp();
      }
      if (t >= 1) {
        const int i = t - 1, sb = i & 1;
        ok = __all_sync(0xffffffffu, ok && mbar_wait(&p_full[sb], (i >> 1) & 1));
        if (!ok) break;
        tc_fence_after();
        for (int i4 = 0; ok && i4 < C::NVB; i4 += C::CPS) {
          const uint32_t vbase = take();   // V blocks i4 ..: 64 keys x 64 CPS output columns, MN-major
          if (!ok) break;
          const uint64_t vd0 = umma_desc_sw128(vbase, C::CHUNK, 1024);
          if (elect_one()) {
#pragma unroll
            for (int ks = 0; ks < C::NK / 16; ++ks)
              umma_ts(tmem + i4 * 64, tmem + C::S_COL0 + sb * 64 + ks * 8, vd0 + static_cast<uint64_t>(ks * 2048 / 16),
                      idO, (i > 0 || ks > 0) ? 1u : 0u);
          }
          __syncwarp();
          give();
        }
        if (elect_one()) umma_commit(&o_bar[i & 1]);   // PV i completes phase i / 2 of o_bar[i & 1]
        __syncwarp();
      }
    }
    if (!ok && lane == 0) atomicOr(p.err, FA_DEV_ERR_TIMEOUT);
    // every MMA the elected lane issued has finished before tensor memory is freed
    if (elect_one()) umma_commit(&done_bar);
    __syncwarp();
    if (!__all_sync(0xffffffffu, mbar_wait(&done_bar, 0)) && lane == 0) atomicOr(p.err, FA_DEV_ERR_TIMEOUT);
  } else {
    // ------------------------------------------------------------- softmax
    // Two warps per row quarter (tensor-memory lane access follows warp % 4):
    // the first four take columns [0, 32) of each 64-key tile, the other four
    // columns [32, 64).  The two halves of a row exchange their tile maxima
    // through shared memory (double buffered by tile parity) once per tile,
    // each rounded up to an integer so that both halves take the same value
    // (any common base gives the same softmax); that barrier ANDs each warp's wait
    // result, so all eight leave the loop together.  Each half keeps its share
    // of the denominator; the shares meet once in the epilogue, through the
    // ring, which is idle by then.
    __shared__ short sm_mx[2][2][C::M];   // [tile parity][half][row]: max_code values
    constexpr int SMX_BAR = 2, SMX_THREADS = C::NSMX * 32;
    const int half = (warp - (C::W_MMA + 1)) >> 2;
    const int quarter = warp & 3;
    bool range_bad = false;
    const int r = quarter * 32 + lane;   // query row = tensor-memory lane
    const int tl = r / p.g, hj = r % p.g;
    const int t = x.t0 + tl;
    const bool row_ok = t < x.n;
    const int qpos = x.P + t;
    const uint32_t trow = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    {
      // this row's first NQT * 64 query values into tensor memory (row =
      // lane, 16-bit pairs per column: the A-operand layout of the S MMA),
      // half h moving blocks h, h + 2, ... out of the staging slots (rows past
      // the last token arrive as zeros).  8-bit slabs: the MMAs run in f16,
      // so those values go as f16, and Q's shared-memory blocks are rewritten
      // in place as f16 too.  Then the staging slots are released.
      bool qok = mbar_wait(qst_full, 0);
      if constexpr (C::Q8) qok = mbar_wait(q_full, 0) && qok;
      if (!__all_sync(0xffffffffu, qok) && lane == 0) atomicOr(p.err, FA_DEV_ERR_TIMEOUT);
      constexpr int QBLK = C::Q8 ? C::KB : C::NQT;
      uint32_t qbig = 0;
#pragma unroll 1
      for (int kb = half; kb < QBLK; kb += 2) {
        uint8_t* blk = kb < C::NQT ? ring + C::QST_OFF + kb * (C::M * 128) : qs + (kb - C::NQT) * (C::M * 128);
        uint32_t w[32];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 v = *reinterpret_cast<const uint4*>(blk + sw128(r, u));
          w[4 * u] = v.x;
          w[4 * u + 1] = v.y;
          w[4 * u + 2] = v.z;
          w[4 * u + 3] = v.w;
        }
        if constexpr (C::Q8) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            qbig |= bf16x2_past_f16(w[i]);
            w[i] = pack_f16x2_sat(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
          }
        }
        if (kb < C::NQT) {
          tmem_st32(trow + C::Q_COL0 + kb * 32, w);
        } else {   // 8-bit slabs only
#pragma unroll
          for (int u = 0; u < 8; ++u)
            *reinterpret_cast<uint4*>(blk + sw128(r, u)) = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
        }
      }
      if constexpr (C::Q8) {
        fence_proxy_async_smem();   // the Q rows written here, for the S MMA
        if (__any_sync(0xffffffffu, qbig != 0) && lane == 0) atomicOr(p.err, FA_DEV_ERR_RANGE);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(qt_full);
        mbar_arrive(q_free);
      }
    }
    const int klo = (p.kind == FA_FULL) ? 0 : qpos - p.window + 1;
    const float sc = p.scale_log2;
    // l_run: this half's share of the denominator, the sum of the rounded
    // weights the PV MMA uses (so constant V gives exactly that constant;
    // 8-bit slabs: of the unrounded weights, the V scale being folded in);
    // l_lse: the sum of the unrounded weights, for lse
    float m_run = -INFINITY, l_run = 0.f, l_lse = 0.f;
    // 8-bit slabs: the exponent base sits 2^7 below the running maximum of
    // score + the half's largest log2 cv, so the weighted P stays below 2^15
    constexpr float MB_OFF = C::Q8 ? 7.0f : 0.0f;
    bool ok = true, bad = false;
    constexpr int OH = C::DS / 2;            // O columns this half rescales and writes
    // 8-bit slabs: per tile the scale slot holds ck (multiplies the raw
    // scores) and cv (multiplies the weights) of the 64 keys, and per half of
    // them the largest log2 cv, which joins the maximum
    for (int j = 0; j < nt; ++j) {
      const int sb = j & 1;
      const uint32_t s_col = C::S_COL0 + sb * 64;
      bool got = mbar_wait(&s_full[sb], (j >> 1) & 1);
      if constexpr (C::Q8) got = mbar_wait(&sc_full[j % C::SCL_R], (j / C::SCL_R) & 1) && got;
      got = __all_sync(0xffffffffu, got);
      const float* sslot = scl + (j % C::SCL_R) * (C::SCL_TILE / 4);
      const float* ck = sslot + 32 * half;   // this half's 32 keys
      const float* cvh = sslot + 64 + 32 * half;
      const bool pre = x.prefix(j);
      const int st0 = x.start(j) + 32 * half;   // key of this half's first column
      // raw scores of this row's visible keys (one interval [clo, chi] per
      // row from the causal, window and prefix-end limits), -inf elsewhere;
      // the scale is applied inside the exponent below
      float sv[32];
      float mt = -INFINITY;
      if (got) {
        tc_fence_after();
        uint32_t sr[32];
        tmem_ld32(trow + s_col + 32 * half, sr);
        tmem_ld_wait();
        const int khi = !row_ok ? -(1 << 30) : (pre ? min(qpos, x.Pk - 1) : qpos);
        const int clo = klo - st0, chi = khi - st0;
        if constexpr (C::Q8) {
          // scaled scores (log2 domain)
          const bool all = __all_sync(0xffffffffu, clo <= 0 && chi >= 31);
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            const float4 k4 = *reinterpret_cast<const float4*>(ck + 4 * c4);
            const float kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int c = 4 * c4 + e;
              const float t = __uint_as_float(sr[c]) * kk[e];
              sv[c] = (all || (c >= clo && c <= chi)) ? t : -INFINITY;
            }
          }
        } else if (__all_sync(0xffffffffu, clo <= 0 && chi >= 31)) {   // all 32 columns visible to the warp's rows
#pragma unroll
          for (int c = 0; c < 32; ++c) sv[c] = __uint_as_float(sr[c]);
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) sv[c] = (c >= clo && c <= chi) ? __uint_as_float(sr[c]) : -INFINITY;
        }
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};   // four chains, then a tree
#pragma unroll
        for (int c = 0; c < 32; ++c) mx[c & 3] = fmaxf(mx[c & 3], sv[c]);
        const float mxa = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
        // 8-bit slabs: plus the half's largest log2 V scale, a bound on
        // score + log2 cv over its keys
        const short mr = max_code(C::Q8 ? mxa + sslot[128 + half] : mxa * sc, range_bad);
        sm_mx[sb][half][r] = mr;
        mt = max_decode(mr);
      }
      // every warp has loaded its S half (so P may now overwrite the S
      // buffer) and published its maximum
      ok = named_bar_and(SMX_BAR, SMX_THREADS, got && !bad);
      if (!ok) break;
      mt = fmaxf(mt, max_decode(sm_mx[sb][half ^ 1][r]));
      const float m_new = fmaxf(m_run, mt);
      const bool need = m_new > m_run + 8.0f;   // rescale only when the max grows by more than 2^8
      if (__any_sync(0xffffffffu, need && m_run > -INFINITY) && j > 0) {
        // PV_{j-1} has finished writing O; this half rescales its O columns
        if (__all_sync(0xffffffffu, mbar_wait(&o_bar[(j - 1) & 1], ((j - 1) >> 1) & 1))) {
          tc_fence_after();
          const float f = (need && m_run > -INFINITY) ? ex2(m_run - m_new) : 1.0f;
#pragma unroll 1
          for (int c = half * OH; c < (half + 1) * OH; c += 32) {
            uint32_t o[32];
            tmem_ld32(trow + c, o);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
            tmem_st32(trow + c, o);
          }
          tmem_st_wait();
        } else {
          bad = true;   // leaves the loop at the next tile's barrier
          if (lane == 0) atomicOr(p.err, FA_DEV_ERR_TIMEOUT);
        }
      }
      if (need) {
        const float f = (m_run > -INFINITY) ? ex2(m_run - m_new) : 0.f;
        l_run *= f;
        l_lse *= f;
        m_run = m_new;
      }
      uint32_t pk[16];
      float ps[4] = {0.f, 0.f, 0.f, 0.f}, pe[2] = {0.f, 0.f};
      // a row with no visible key so far has m_run = -inf and only -inf scores: exponent base 0 gives 0
      const float mb = (m_run > -INFINITY) ? m_run - MB_OFF : 0.f;
      if constexpr (C::Q8) {
        // weight q = 2^(score - mb) into the denominator; q x cv, below 2^15
        // (score + log2 cv <= m_run + 8), into the PV MMA as f16
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 v4 = *reinterpret_cast<const float4*>(cvh + 4 * c4);
          const float q0 = ex2(sv[4 * c4] - mb), q1 = ex2(sv[4 * c4 + 1] - mb);
          const float q2 = ex2(sv[4 * c4 + 2] - mb), q3 = ex2(sv[4 * c4 + 3] - mb);
          pe[0] += q0 + q1;
          pe[1] += q2 + q3;
          pk[2 * c4] = pack_f16x2(q0 * v4.x, q1 * v4.y);
          pk[2 * c4 + 1] = pack_f16x2(q2 * v4.z, q3 * v4.w);
        }
        l_run += pe[0] + pe[1];
      } else {
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const float p0 = ex2(fmaf(sv[2 * c], sc, -mb));
          const float p1 = ex2(fmaf(sv[2 * c + 1], sc, -mb));
          pe[c & 1] += p0 + p1;
          // the denominator sums the rounded weights the PV MMA uses
          pk[c] = pack_bf16x2(p0, p1);
          ps[c & 3] += __uint_as_float(pk[c] << 16) + __uint_as_float(pk[c] & 0xffff0000u);
        }
        l_run += (ps[0] + ps[1]) + (ps[2] + ps[3]);
      }
      l_lse += pe[0] + pe[1];
      tmem_st16(trow + s_col + 16 * half, pk);   // P of keys [32 half, 32 half + 32): 16 columns of 16-bit pairs
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&p_full[sb]);
        if constexpr (C::Q8) mbar_arrive(&sc_empty[j % C::SCL_R]);   // this tile's scales are read
      }
    }
    // ------------------------------------------------------------ epilogue
    if (__any_sync(0xffffffffu, range_bad) && lane == 0) atomicOr(p.err, FA_DEV_ERR_RANGE);
    bool fin = ok;
    if (fin && nt > 0) fin = __all_sync(0xffffffffu, mbar_wait(&o_bar[(nt - 1) & 1], ((nt - 1) >> 1) & 1));
    // every MMA has completed, so every ring slot was consumed: the ring is idle
    float* sm_l = reinterpret_cast<float*>(ring);   // [half][row]: rounded sums, then unrounded ones
    if (fin) {
      sm_l[half * C::M + r] = l_run;
      sm_l[(2 + half) * C::M + r] = l_lse;
    }
    fin = named_bar_and(SMX_BAR, SMX_THREADS, fin);
    const float l_tot = fin ? l_run + sm_l[(half ^ 1) * C::M + r] : 0.f;
    const float l_all = fin ? l_lse + sm_l[(2 + (half ^ 1)) * C::M + r] : 0.f;
    if (!fin && lane == 0) atomicOr(p.err, FA_DEV_ERR_TIMEOUT);
    // The output rows leave through the idle ring: each lane puts its row's
    // 128 bf16 columns (256 bytes; rows 272 bytes apart, so the 16-byte
    // stores are free of bank conflicts) into its warp's part, then copies
    // the row out with one bulk copy (plain stores left the SM at about 16
    // bytes per cycle, ~2 us per CTA).
    auto stage = [&](int c, const uint32_t (&w)[16]) {   // columns [c, c + 32) of this half
      uint8_t* stg = ring + 4096 + (quarter * 2 + half) * (32 * 272) + lane * 272;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        *reinterpret_cast<uint4*>(stg + ((c >> 5) * 4 + e) * 16) = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
    };
    auto write_rows = [&]() {
      const uint8_t* stg = ring + 4096 + (quarter * 2 + half) * (32 * 272) + lane * 272;
      fence_proxy_async_smem();   // the rows just written, for the bulk copy's reads
      if (row_ok) bulk_store(p.out + (static_cast<size_t>(x.qo0 + t) * p.Hq + x.h * p.g + hj) * D + x.ds * C::DS + half * OH,
                             stg, OH * 2);
      bulk_store_drain();
    };
    if (x.ks == 2) {
      // A split job: leave this CTA's partial (unnormalised O over its tiles,
      // the exponent base and both sums) in the workspace, then arrive; the
      // second arrival combines the two on a common base.  Each lane moves
      // whole 16-byte pieces of its row, laid out so that a warp's 32 lanes
      // touch 512 consecutive bytes.  A CTA that timed out still arrives, so
      // the counter is left zero (its error bit says the output is void).
      // The arrival result is shared through the idle ring, past the sums (a
      // static shared variable would take the kernel past its shared-memory
      // budget at head_dim 512).
      volatile int& sh_last = *reinterpret_cast<volatile int*>(ring + 4 * C::M * sizeof(float));
      const float base = (m_run > -INFINITY) ? m_run - MB_OFF : -INFINITY;
      const size_t pj = static_cast<size_t>(x.slot) * 2;
      const size_t grp = static_cast<size_t>(quarter * 2 + half) * 32;   // this warp's float4 columns
      if (fin) {
        float4* po = p.ws_o + (pj + x.s) * (C::M * C::DS / 4) + grp * 32 + lane;
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < OH; c += 32) {
          uint32_t o[32];
          tmem_ld32(trow + half * OH + c, o);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 8; ++e)
            po[(c / 4 + e) * 32] = make_float4(__uint_as_float(o[4 * e]), __uint_as_float(o[4 * e + 1]),
                                               __uint_as_float(o[4 * e + 2]), __uint_as_float(o[4 * e + 3]));
        }
        if (half == 0) p.ws_ml[(pj + x.s) * C::M + r] = make_float4(base, l_tot, l_all, 0.f);
      }
      // the barrier orders every lane's partial writes before the release /
      // acquire add, which publishes them and, for the second arrival, makes
      // the other CTA's partial visible
      named_bar_sync(SMX_BAR, SMX_THREADS);
      if (warp == C::W_MMA + 1 && lane == 0) {
        const int old = atom_add_acq_rel_gpu(p.ws_cnt + x.slot, 1);
        int last = 0;
        if (old == 1) {
          last = 1;
          atomicExch(p.ws_cnt + x.slot, 0);   // zero for the next launch
        } else if (old != 0) {
          atomicOr(p.err, FA_DEV_ERR_WORKSPACE);
        }
        sh_last = last;
      }
      named_bar_sync(SMX_BAR, SMX_THREADS);
      if (sh_last && fin) {
        // the combination is written in the CTAs' split order (first half of
        // the tiles, then second), not in arrival order, so the result does
        // not depend on which CTA finished last
        const float4 om = __ldcg(p.ws_ml + (pj + (x.s ^ 1)) * C::M + r);
        const bool first = x.s == 0;
        const float b0 = first ? base : om.x, b1 = first ? om.x : base;
        const float bm = fmaxf(b0, b1);
        const float f0 = (b0 > -INFINITY) ? ex2(b0 - bm) : 0.f;
        const float f1 = (b1 > -INFINITY) ? ex2(b1 - bm) : 0.f;
        const float lt = (first ? l_tot : om.y) * f0 + (first ? om.y : l_tot) * f1;
        const float la = (first ? l_all : om.z) * f0 + (first ? om.z : l_all) * f1;
        const float inv = (lt > 0.f) ? 1.0f / lt : 0.f;
        const float w0 = f0 * inv, w1 = f1 * inv;
        const float4* oo = p.ws_o + (pj + (x.s ^ 1)) * (C::M * C::DS / 4) + grp * 32 + lane;
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < OH; c += 32) {
          uint32_t o[32];
          tmem_ld32(trow + half * OH + c, o);
          tmem_ld_wait();
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float4 v = __ldcg(oo + (c / 4 + e) * 32);
            const float oth[4] = {v.x, v.y, v.z, v.w};
            float y[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float own = __uint_as_float(o[4 * e + k]);
              y[k] = (first ? own : oth[k]) * w0 + (first ? oth[k] : own) * w1;
            }
            w[2 * e] = pack_bf16x2(y[0], y[1]);
            w[2 * e + 1] = pack_bf16x2(y[2], y[3]);
          }
          stage(c, w);
        }
        write_rows();
        if (row_ok && half == 0 && x.ds == 0 && p.lse)
          p.lse[static_cast<size_t>(x.qo0 + t) * p.Hq + x.h * p.g + hj] =
              (bm > -INFINITY && la > 0.f) ? (bm + __log2f(la)) * 0.69314718055994531f : -INFINITY;
      }
    } else if (fin) {
      tc_fence_after();
      const float inv = (l_tot > 0.f) ? 1.0f / l_tot : 0.f;
#pragma unroll 1
      for (int c = 0; c < OH; c += 32) {
        uint32_t o[32];
        tmem_ld32(trow + half * OH + c, o);
        tmem_ld_wait();
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          w[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
        stage(c, w);
      }
      write_rows();
      if (row_ok && half == 0 && x.ds == 0 && p.lse)
        p.lse[static_cast<size_t>(x.qo0 + t) * p.Hq + x.h * p.g + hj] =
            (m_run > -INFINITY && l_all > 0.f) ? (m_run - MB_OFF + __log2f(l_all)) * 0.69314718055994531f : -INFINITY;
    }
  }

  // ------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == C::W_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D, int KV>
static cudaError_t launch_extend_t(const ExtendArgs& a, const ExtK& k, cudaStream_t s) {
  using C = ExtCfg<D, KV>;
  static unsigned int done = 0;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(extend_kernel<D, KV>), C::SMEM_ALLOC, &done);
  if (e != cudaSuccess) return e;
  const long long jobs = static_cast<long long>(k.gx) * k.gy * a.B;
  const long long ctas = k.split_from + 2 * (jobs - k.split_from);
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  return launch_pdl(extend_kernel<D, KV>, dim3(static_cast<unsigned>(ctas)), dim3(C::NTHR), C::SMEM_ALLOC, s, a.tm_q,
                    *a.tm_k, *a.tm_v, a.tm_kx, a.tm_vx, k);
}

// The jobs (from the end of the launch order) that run as two CTAs each.
// One CTA fits an SM, so a launch of J equal jobs takes ceil(J / SMs) job
// times; when its last wave is at most half full, splitting that wave's jobs
// in two (so every SM has at most half a job left) saves up to half a job
// time, less the partials' write and merge, which long jobs (8 key tiles or
// more, estimated from the length bounds) amortise.
static int split_jobs(const ExtendArgs& a, long long jobs) {
  if (!a.split_ws || a.split_mode == 0 || jobs <= 0) return 0;
  if (a.split_mode == 2) return static_cast<int>(jobs < a.split_cap ? jobs : a.split_cap);
  const long long sms = sm_count();
  const long long tail = jobs % sms;
  const long long keys = (a.kind == FA_SLIDING ? std::min(a.max_prefix_len, a.window) : a.max_prefix_len) +
                         a.max_q_len / 2;
  if (tail == 0 || 2 * tail > sms || keys < 8 * 64 || tail > a.split_cap) return 0;
  return static_cast<int>(tail);
}

cudaError_t launch_extend(const ExtendArgs& a, cudaStream_t s) {
  ExtK k{};
  k.q = static_cast<const __nv_bfloat16*>(a.q);
  k.k_slab = static_cast<const uint8_t*>(a.k_slab);
  k.v_slab = static_cast<const uint8_t*>(a.v_slab);
  k.k_scale = a.k_scale;
  k.v_scale = a.v_scale;
  k.k_ext = static_cast<const uint8_t*>(a.k_ext);
  k.v_ext = static_cast<const uint8_t*>(a.v_ext);
  k.num_tokens = a.num_tokens;
  k.qo_indptr = a.qo_indptr;
  k.prefix_lens = a.prefix_lens;
  k.seq_lens = a.seq_lens;
  k.keys_in_pages = a.keys_in_pages;
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
  k.dslices = a.D / ExtCfg<256>::DS;
  k.early_metadata = a.early_metadata;
  k.scale_log2 = a.sm_scale * 1.4426950408889634f;
  k.gx = (a.max_q_len + k.T - 1) / k.T;
  k.gy = a.Hkv * k.dslices;
  const long long jobs = static_cast<long long>(k.gx) * k.gy * a.B;
  if (jobs > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const int nsplit = split_jobs(a, jobs);
  k.split_from = static_cast<int>(jobs - nsplit);
  if (nsplit > 0) {
    const ExtSplitLayout l = ext_split_layout(a.split_cap);
    uint8_t* ws = static_cast<uint8_t*>(a.split_ws);
    k.ws_cnt = reinterpret_cast<int*>(ws);
    k.ws_ml = reinterpret_cast<float4*>(ws + l.off_ml);
    k.ws_o = reinterpret_cast<float4*>(ws + l.off_o);
  }
  if (a.kv_dtype == FA_KV_INT8)
    return a.D == 256 ? launch_extend_t<256, FA_KV_INT8>(a, k, s) : launch_extend_t<512, FA_KV_INT8>(a, k, s);
  if (a.kv_dtype == FA_KV_FP8)
    return a.D == 256 ? launch_extend_t<256, FA_KV_FP8>(a, k, s) : launch_extend_t<512, FA_KV_FP8>(a, k, s);
  return a.D == 256 ? launch_extend_t<256, FA_KV_BF16>(a, k, s) : launch_extend_t<512, FA_KV_BF16>(a, k, s);
}

}  // namespace fa
