/*
 * fa.h -- C ABI of the GB300 (sm_103a) paged-KV attention library.
 *
 * Gemma-4-style attention over a block-table KV cache with two per-layer
 * regimes and KV sharing:
 *
 *   full layers     purely causal, kv_pos <= q_pos, head_dim 512;
 *   sliding layers  causal and q_pos - kv_pos < W, head_dim 256, where W
 *                   counts the current token (W = 1024 sees 1023 earlier
 *                   positions; a FlashInfer-style inclusive window_left is
 *                   W - 1).
 *                   ["unsloth gemma4_flex_inference.py" commit history,
 *                    commit "block mask per attention regime";
 *                    "pegainfer issue #807", Description, second paragraph]
 *
 *   KV-shared layers own no slab: they read the slab (and, in the 8-bit
 *   formats, the scales) of their source, the last earlier owning layer of the
 *   same attention type, and the store skips them.
 *                   ["FreeToken PR #898: read the source layer's kv slab on
 *                    kv-shared layers", description bullets;
 *                    "unsloth commit dee9371", commit message]
 *
 * Conventions shared by every call
 * --------------------------------
 * - Ownership.  The caller allocates and owns every device buffer (slabs,
 *   scales, q/k/v, tables, outputs, workspace) and every stream.  The library
 *   owns only the host-side descriptor returned by fa_cache_create.  No call
 *   allocates or frees device memory.
 * - Streams.  `stream` is a cudaStream_t handle passed as void*; NULL is the
 *   legacy default stream.  Device work is enqueued asynchronously; a call
 *   returns after host-side validation and the launches.
 * - Errors.  Every call returns an fa_status.  Host-side validation failures
 *   return without launching anything; fa_last_error() gives a message
 *   (thread-local).  Launch failures return FA_ERR_CUDA.  Faults that only the
 *   device can see (a page id outside [0, num_pages), a slot outside the pool,
 *   a sequence longer than the bound the caller promised, a bounded wait that
 *   ran out) never trap: the kernel skips the access, sets a bit in the
 *   cache's device error word and finishes; fa_get_device_error() reads and
 *   clears it.  Each live cache has a word of its own (a slot of a fixed
 *   device array of FA_MAX_CACHES words, one array per device), so calls on
 *   one cache never see or clear another cache's errors.
 * - Types.  bf16 tensors are IEEE bfloat16 (2 bytes); int32 tables are
 *   little-endian int32_t; all tensors are dense row-major with the shapes
 *   given below.  Device pointers must be 16-byte aligned.
 * - GQA.  Query head j reads KV head j / (Hq / Hkv); Hq must be a multiple of
 *   Hkv.  (The pages do not state the mapping; contiguous groups are the
 *   usual repeat-kv convention.)
 *
 * Physical layouts (chosen by this library; results depend only on the
 * logical rows, so any physical page order gives the same attention output):
 *   bf16 slab     K, V: bf16 [num_pages][Hkv][page_size][D]
 *   int8 slab     K, V: int8 [num_pages][Hkv][page_size][D]  (codes)
 *                 k_scale, v_scale: float [num_pages][Hkv][page_size]
 *   fp8 slab      K, V: uint8 [num_pages][Hkv][page_size][D]  (e4m3 codes)
 *                 k_scale, v_scale: float [num_pages][Hkv][page_size]
 *   slot          page * page_size + offset; logical position p of sequence b
 *                 lives in page block_table[b][p / page_size], offset
 *                 p % page_size.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(FA_BUILD) && defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned pointer ... */
  FA_ERR_UNSUPPORTED = 2,   /* a layout the method refuses or the library does not implement */
  FA_ERR_NOT_BOUND = 3,     /* the layer's slab owner has no slab bound yet   */
  FA_ERR_WORKSPACE = 4,     /* workspace smaller than fa_decode_workspace_bytes */
  FA_ERR_CUDA = 5,          /* a CUDA runtime call or launch failed           */
  FA_ERR_DEVICE = 6         /* reserved for device-side error reports         */
} fa_status;

/* KV slab formats.  The 8-bit per-token-head formats ("FreeToken PR #898",
 * description: int8_per_token_head and fp8_per_token_head, a shared layer
 * reading its source's scales) hold one code byte per element and one fp32
 * scale per (token, KV head), separately for K and V; the value is
 * code * scale.  fp8 codes are e4m3 (the OCP 8-bit floating point E4M3
 * encoding without infinities, largest finite magnitude 448). */
typedef enum { FA_KV_BF16 = 0, FA_KV_INT8 = 1, FA_KV_FP8 = 2 } fa_kv_dtype;
typedef enum { FA_FULL = 0, FA_SLIDING = 1 } fa_layer_kind;

/* kv_source values besides an explicit earlier layer index */
#define FA_KV_OWN (-1)    /* the layer owns a slab */
#define FA_KV_AUTO (-2)   /* shared: source = last earlier owning layer of its kind */

/* Device error bits reported by fa_get_device_error */
#define FA_DEV_ERR_PAGE 0x1u       /* a visible page id was outside [0, num_pages) */
#define FA_DEV_ERR_SLOT 0x2u       /* a store slot was >= num_pages * page_size    */
#define FA_DEV_ERR_BOUND 0x4u      /* a length exceeded the caller's max bound      */
#define FA_DEV_ERR_TIMEOUT 0x8u    /* a bounded barrier wait ran out                */
#define FA_DEV_ERR_WORKSPACE 0x10u /* decode or extend-split workspace counters
                                      were not zero                                 */
#define FA_DEV_ERR_RANGE 0x20u     /* a value out of the kernels' range: an f16
                                      operand saturated (8-bit formats: a q, or
                                      an extend k_ext / v_ext, magnitude of 65520
                                      or more), or an extend score with
                                      |sm_scale * q.k| * log2(e) of 32767 or
                                      more                                          */

/* Most fa_cache descriptors that may be live at once (each holds one device
 * error word). */
#define FA_MAX_CACHES 4096

/* One attention layer.  kind: fa_layer_kind.  head_dim: 256 or 512 (other
 * widths return FA_ERR_UNSUPPORTED; the pages name exactly these two).
 * window: Gemma's W for sliding layers (>= 1, counts the current token);
 * ignored for full layers.  kv_source: FA_KV_OWN, FA_KV_AUTO, or an explicit
 * earlier owning layer of the same kind and KV geometry.  sm_scale: the
 * softmax scale applied to q.k (usually 1/sqrt(head_dim)). */
typedef struct {
  int32_t kind;
  int32_t head_dim;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t window;
  int32_t kv_source;
  float sm_scale;
} fa_layer_desc;

typedef struct fa_cache fa_cache;   /* opaque host-side descriptor */

/* Build the layer -> slab map for n_layers layers sharing one page pool of
 * num_pages pages of page_size tokens, in kv_dtype.  Resolves every shared
 * layer's source by the rule of "FreeToken PR #898" (description, first
 * bullet: the last earlier layer of its attention type) and refuses, with
 * FA_ERR_UNSUPPORTED, a shared layer that has no earlier owning layer of its
 * kind, a source that is itself shared or of another kind, or a source whose
 * head_dim / num_kv_heads differ (review thread of the same PR: such a
 * layout is refused, not served).  page_size must be a multiple of 16 and at
 * most 256.  On success *out receives a descriptor to free with
 * fa_cache_destroy.  At most FA_MAX_CACHES descriptors may be live at once
 * (FA_ERR_UNSUPPORTED beyond).  Host only; no CUDA call. */
FA_API fa_status fa_cache_create(const fa_layer_desc* layers, int32_t n_layers, int32_t num_pages,
                          int32_t page_size, int32_t kv_dtype, fa_cache** out);

/* Free the descriptor (NULL is accepted).  Device buffers stay the caller's. */
FA_API void fa_cache_destroy(fa_cache* cache);

/* Cache flags (fa_cache_set_flags). */
#define FA_FLAG_EARLY_METADATA 0x1u
#define FA_FLAG_EXTEND_SPLIT_ALL 0x2u

/* Set FA_FLAG_* options for every later call on this cache (default 0).
 * FA_FLAG_EARLY_METADATA: the caller guarantees that the index arrays of each
 * call (block_table, seq_lens, slot_mapping, qo_indptr, prefix_lens) are
 * final when the call is enqueued and are not written by the kernel launched
 * immediately before it on the same stream (the usual case when they are
 * copied from the host).  The kernels, which launch with programmatic
 * dependent launch, then read them while that kernel is still finishing, and
 * wait for it only before touching q, k, v, the slabs and the outputs.
 * Without the flag every read waits.
 * FA_FLAG_EXTEND_SPLIT_ALL: with an extend workspace bound
 * (fa_cache_bind_extend_workspace), split as many jobs of every extend and
 * multi-token decode launch as it holds, whatever their size (the merge is
 * then exercised on any input; slower in general).
 * Unknown bits: FA_ERR_INVALID_ARG.  No counterpart on the pages: these are
 * launch options of this library.  Host only. */
FA_API fa_status fa_cache_set_flags(fa_cache* cache, uint32_t flags);

/* Bytes of the extend split workspace on the current device (about 20 MB on
 * 152 SMs).  The extend kernel runs one CTA per SM, one per job (a 128-row
 * block of one sequence's queries, one KV head, one 256-column output
 * slice), all jobs of a launch about equally long on uniform inputs; when a
 * launch's last wave would leave more than half of the SMs idle, the jobs of
 * that wave can each run as two CTAs over the two halves of their key tiles,
 * merged on a common softmax base by the second to finish.  The workspace
 * holds those jobs' partials (half the SM count of jobs).  No counterpart on
 * the pages: a scheduling option of this library.  Host only. */
FA_API size_t fa_extend_workspace_bytes(void);

/* Let extend (fa_paged_extend_attn) and multi-token decode
 * (fa_paged_decode_multi_attn) calls on `cache` split their last wave as
 * described above, through `workspace`: device memory of the current device,
 * 256-byte aligned, of `bytes` >= the partials of one job (fewer than
 * fa_extend_workspace_bytes() bytes holds fewer jobs).  The caller keeps
 * ownership; it must stay allocated while calls may use it, and calls on
 * the cache that use it must run in stream order (one stream, or streams
 * ordered by events): concurrent calls would share its slots.  Zeroes its
 * arrival counters (synchronous); each launch leaves them zero.  A launch
 * splits when the wave is at most half full and its length bounds promise
 * 8 key tiles (512 keys) or more per job.  NULL unbinds.  Errors: FA_ERR_INVALID_ARG
 * (misaligned), FA_ERR_WORKSPACE (too small for one job), FA_ERR_CUDA. */
FA_API fa_status fa_cache_bind_extend_workspace(fa_cache* cache, void* workspace, size_t bytes);

/* Give the sliding layers' slabs a page pool of their own (the pages' window
 * pool: "FreeToken PR #898", description, the window slots come from one
 * full-to-window index mapping; "pegainfer issue #807", Description, the
 * sliding group releases pages the full group still reads).  Sliding layers
 * then hold window_pages pages each (full layers keep num_pages) and their
 * block tables index that pool: entries for positions outside the window
 * may be -1 or point at pages since reused, as no kernel reads them.  A page
 * id >= window_pages in a sliding layer's table sets FA_DEV_ERR_PAGE.  Call
 * before binding any sliding slab; 0 restores the single pool. */
FA_API fa_status fa_cache_set_window_pool(fa_cache* cache, int32_t window_pages);

/* Slab owner of `layer`: the layer itself if it owns a slab, else its
 * resolved source.  Host only. */
FA_API fa_status fa_cache_layer_source(const fa_cache* cache, int32_t layer, int32_t* slab_owner);

/* Bytes the caller must allocate for one of K or V of an owning layer
 * (num_pages * Hkv * page_size * D * elem) and for one of k_scale or v_scale
 * (0 in bf16).  A shared layer reports 0 and 0.  Host only. */
FA_API fa_status fa_cache_slab_bytes(const fa_cache* cache, int32_t layer, size_t* kv_bytes,
                              size_t* scale_bytes);

/* Bind caller-owned device buffers as the slab of an owning layer (k, v in the
 * layout above; k_scale, v_scale required in the 8-bit formats, ignored in
 * bf16).  Binding a shared layer returns FA_ERR_INVALID_ARG: it reads its
 * source's slab.  Rebinding replaces the previous pointers.  Encodes the TMA
 * descriptors the kernels use and clears the cache's device error word on
 * the current device (synchronously: do not call it during stream capture),
 * so it needs a CUDA device (FA_ERR_CUDA when the driver cannot be
 * reached). */
FA_API fa_status fa_cache_bind_slab(fa_cache* cache, int32_t layer, void* k, void* v, float* k_scale,
                             float* v_scale);

/* Bytes one token costs across the slabs of the owning layers of `kind`
 * (fa_layer_kind): per owning layer and KV head 2 * (D * elem + scale bytes).
 * Shared layers cost nothing ("FreeToken PR #898", description bullet on
 * kv_cache_group_specs; its "End to end" section prints these unit_bytes).
 * Host only. */
FA_API size_t fa_kv_bytes_per_token(const fa_cache* cache, int32_t kind);

/* Paged KV store ("FreeToken PR #898", description bullet on HybridSWAKVCache
 * and store_kv; "unsloth commit dee9371": the store layer writes its
 * post-rotary k, v into its paged cache).
 * k, v: bf16 [T][Hkv][D] post-RoPE rows of T new tokens (device).
 * slot_mapping: int32 [T] (device); token t goes to slot slot_mapping[t];
 * a negative slot is padding and is skipped; a slot >= num_pages * page_size
 * is skipped and sets FA_DEV_ERR_SLOT.
 * bf16 format: a bit-exact copy.  int8 format: per (token, head), separately
 * for K and V, a = max|x| in fp32, s = a / 127 (IEEE division), codes
 * c = clamp(rint(x / s), -127, 127) with rint rounding half to even; a = 0
 * gives s = 0 and all-zero codes.  fp8 format: the same with s = a / 448
 * and codes the e4m3 value nearest to the fp32 quotient x / s (ties to the
 * even mantissa, magnitudes above 448 saturating to 448, sign kept); a = 0
 * gives s = 0 and all-zero codes.
 * A KV-shared layer stores nothing: FA_OK, no launch.  T == 0: FA_OK, no
 * launch. */
FA_API fa_status fa_kv_store(fa_cache* cache, int32_t layer, const void* k, const void* v,
                      const int32_t* slot_mapping, int32_t T, void* stream);

/* Workspace bytes fa_paged_decode_attn needs for this layer, batch and bound
 * on the sequence lengths: one arrival counter per (sequence, KV head, group
 * of up to 8 query heads) followed by the split-K partial rows.  0 when a
 * single CTA serves the whole call.  Host only. */
FA_API size_t fa_decode_workspace_bytes(const fa_cache* cache, int32_t layer, int32_t B,
                                 int32_t max_seq_len);

/* Paged decode attention, one new token per sequence (split-K online softmax,
 * GQA-packed so each KV page is read once for all Hq / Hkv query heads).
 * q: bf16 [B][Hq][D] (device).  block_table: int32 [B][max_pages_per_seq].
 * seq_lens: int32 [B], the context length INCLUDING the current token, whose
 * k, v must already be stored; the query sits at q_pos = seq_lens[b] - 1.
 * Full layers attend to positions [0, q_pos]; sliding layers to
 * [max(0, q_pos - W + 1), q_pos] and read only the pages that hold them, so
 * block-table entries outside the window may be -1 (never read).
 * A shared layer reads its source's slab and scales.
 * max_seq_len: host bound on every seq_lens[b] (longer ones set
 * FA_DEV_ERR_BOUND and are cut at the bound).
 * out: bf16 [B][Hq][D].  lse: optional float [B][Hq], natural-log
 * sum-exp of the scaled scores.  seq_lens[b] <= 0 gives out = 0 and
 * lse = -inf.  Over 8-bit slabs q is converted to f16 for the tensor cores:
 * an element of magnitude 65536 or more saturates to +-65504 and sets
 * FA_DEV_ERR_RANGE.  workspace: device scratch of at least
 * fa_decode_workspace_bytes(cache, layer, B, max_seq_len) bytes (may be NULL
 * when that is 0), 256-byte aligned.  Zero it once before its first use: its
 * leading counters must start at zero, and every call that completes leaves
 * them zero again, so the same buffer serves later calls on the same stream
 * without clearing.  Calls that run concurrently must not share a workspace.
 * After a call that reported FA_DEV_ERR_TIMEOUT, zero it again (a counter
 * found non-zero sets FA_DEV_ERR_WORKSPACE).  Reference: "unsloth commit
 * dee9371" (shared layers read the source's paged cache on decode) and the
 * regimes above. */
FA_API fa_status fa_paged_decode_attn(fa_cache* cache, int32_t layer, const void* q,
                               const int32_t* block_table, int32_t max_pages_per_seq,
                               const int32_t* seq_lens, int32_t B, int32_t max_seq_len,
                               void* out, float* lse, void* workspace, size_t workspace_bytes,
                               void* stream);

/* Store and decode in one launch: the effect of fa_kv_store(cache, layer,
 * k_new, v_new, slot_mapping, B) followed by fa_paged_decode_attn with the
 * same remaining arguments, for an owning layer, without a second kernel on
 * the dependency chain of the step ("FreeToken PR #898", description: each
 * owning layer stores its rows, then attends; the pages order store before
 * attend).  k_new, v_new: bf16 [B][Hkv][D], the current token's post-RoPE
 * rows (device, 16-byte aligned); slot_mapping: int32 [B], the slot of
 * position seq_lens[b] - 1 (negative: not stored; past the pool: not stored,
 * FA_DEV_ERR_SLOT).  The slot must be the one the block table gives for that
 * position, as with the two separate calls.  Rows are stored in the slab's
 * format (bf16 copy, or the 8-bit quantisation of fa_kv_store, bit for bit)
 * by the CTA that reads the tile holding that position, before it reads it;
 * sequences with seq_lens[b] <= 0 still get their row stored.  For a shared
 * layer k_new, v_new and slot_mapping are ignored (may be NULL) and the call
 * is fa_paged_decode_attn.  Workspace, outputs and errors as
 * fa_paged_decode_attn. */
FA_API fa_status fa_paged_decode_store_attn(fa_cache* cache, int32_t layer, const void* q,
                                     const void* k_new, const void* v_new,
                                     const int32_t* slot_mapping, const int32_t* block_table,
                                     int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t B,
                                     int32_t max_seq_len, void* out, float* lse, void* workspace,
                                     size_t workspace_bytes, void* stream);

/* Most layers one multi-layer store or decode call takes. */
#define FA_MAX_LAYERS_PER_LAUNCH 16

/* The stores of n layers in one launch: the effect of fa_kv_store(cache,
 * layers[i], k[i], v[i], slot_mapping[i], T) for i = 0 .. n - 1 (host arrays
 * of n device pointers; shared layers are skipped, layers of both head_dims
 * may be mixed).  1 <= n <= FA_MAX_LAYERS_PER_LAUNCH; the layers must be
 * distinct owning or shared layers of the cache.  Every row of every layer
 * is stored before the call's stream moves on, so decode calls that follow
 * see all of them. */
FA_API fa_status fa_kv_store_layers(fa_cache* cache, int32_t n, const int32_t* layers, const void* const* k,
                                    const void* const* v, const int32_t* const* slot_mapping, int32_t T,
                                    void* stream);

/* Workspace bytes fa_paged_decode_attn_layers needs: the per-layer
 * workspaces of the n layers laid end to end (each 256-byte aligned).  0 on
 * invalid arguments.  Host only. */
FA_API size_t fa_decode_layers_workspace_bytes(const fa_cache* cache, int32_t n, const int32_t* layers,
                                               int32_t B, int32_t max_seq_len);

/* Paged decode attention of n layers in one launch: the same result per
 * layer, bit for bit, as fa_paged_decode_attn on that layer, with one launch
 * ramp and one tail for all of them instead of one each.  For callers that have the queries of
 * several layers at once: a step that decodes several independent layer
 * stacks, or a benchmark of the attention of a whole step.  The layers must
 * share head_dim and the cache's KV format (a full and a sliding group take
 * two calls) and be distinct; shared layers read their source's slab, so
 * the current token's rows must already be stored (fa_kv_store or
 * fa_kv_store_layers; there is no fused store here).  q, block_table, out,
 * lse: host arrays of n device pointers, per layer as in
 * fa_paged_decode_attn (lse[i] may be NULL; lse itself may be NULL for no
 * lse at all).  seq_lens, B, max_seq_len and max_pages_per_seq are common to
 * all layers.  workspace: at least fa_decode_layers_workspace_bytes bytes,
 * 256-byte aligned, zeroed once, left zero by every completed call (as for
 * fa_paged_decode_attn).  1 <= n <= FA_MAX_LAYERS_PER_LAUNCH. */
FA_API fa_status fa_paged_decode_attn_layers(fa_cache* cache, int32_t n, const int32_t* layers,
                                             const void* const* q, const int32_t* const* block_table,
                                             int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t B,
                                             int32_t max_seq_len, void* const* out, float* const* lse,
                                             void* workspace, size_t workspace_bytes, void* stream);

/* Largest scratch the allocation-free decode below can use (bytes). */
#define FA_NOALLOC_SCRATCH_BYTES (8u << 20)

/* Allocation-free paged decode attention.  The paper has no counterpart: this
 * entry point exists for callers that cannot allocate device memory, such as
 * a plugin inside a serving framework that hands out no allocator, or an
 * engine that reserves its whole memory budget at start-up and forbids
 * cudaMalloc afterwards (it can block or synchronise the device on the hot
 * path).  It computes exactly what fa_paged_decode_attn computes, with the
 * same arguments minus the workspace: its scratch is a fixed array of
 * FA_NOALLOC_SCRATCH_BYTES compiled into the library, which every GPU that
 * loads the library keeps until the process exits.
 * - Limit: a call whose fa_decode_workspace_bytes(cache, layer, B,
 *   max_seq_len) exceeds FA_NOALLOC_SCRATCH_BYTES returns FA_ERR_WORKSPACE and
 *   launches nothing (8 MiB covers, e.g., a batch of 128 at head_dim 512).
 * - Set-up: the first call on each device looks up the array's device address
 *   (with that device current); make that first call before any CUDA-graph
 *   stream capture.
 * - Sharing: every call uses the same array.  Each call clears the counters
 *   it needs before launching, but calls whose work overlaps on the GPU
 *   (different streams, or different threads without ordering) race on the
 *   array and produce wrong results; serialise them.
 * - No cudaMalloc, cudaFree or other allocating routine is called. */
FA_API fa_status fa_paged_decode_attn_noalloc(fa_cache* cache, int32_t layer, const void* q,
                                             const int32_t* block_table, int32_t max_pages_per_seq,
                                             const int32_t* seq_lens, int32_t B, int32_t max_seq_len,
                                             void* out, float* lse, void* stream);

/* Chunked-prefill / extend attention ("FreeToken PR #898", description: the
 * extend kernel takes the prefix from the slab and the current chunk from
 * k_extend / v_extend; "pegainfer issue #807": the prefill chunk size is a
 * capacity parameter).  Sequence b has prefix_lens[b] = P_b tokens already
 * in the cache and n_b = qo_indptr[b+1] - qo_indptr[b] new tokens; new token
 * i sits at position P_b + i and attends to prefix positions (from the slab;
 * in the 8-bit formats code * scale) and chunk positions P_b + j, j <= i
 * (from k_ext / v_ext, bf16, never quantised), under the layer's mask.  Over
 * 8-bit slabs every tensor-core operand is f16 with fp32 accumulation: q,
 * the chunk k, v, the prefix codes (exact in f16), and the softmax weights
 * times the keys' V scales; the K scales multiply the fp32 scores.  Range: a
 * q, k_ext or v_ext element of magnitude 65536 or more (bf16 has nothing
 * between 65280 and 65536, f16 nothing past 65504) saturates to +-65504 and
 * sets FA_DEV_ERR_RANGE; the output is then not the exact attention.  Stored
 * prefix rows have no such limit, and their small magnitudes keep full
 * relative accuracy; chunk values below f16's smallest normal (6.1e-5) are
 * kept as f16 subnormals in steps of 2^-24.  Every slab format: a scaled score |sm_scale * q.k|
 * of 32767 / log2(e) (about 22700) or more is out of range (FA_DEV_ERR_RANGE;
 * the two softmax halves of a row agree on an integer base, kept in 16 bits).
 * q: bf16 [N][Hq][D], k_ext, v_ext: bf16 [N][Hkv][D] with N = qo_indptr[B]
 * (for a shared layer: the source layer's current k, v).  qo_indptr: int32
 * [B+1], non-decreasing, qo_indptr[0] = 0.  num_tokens: the rows of q, k_ext,
 * v_ext and out (qo_indptr[B]; the kernels never read past it).
 * prefix_lens: int32 [B].
 * max_q_len >= every n_b, max_prefix_len >= every P_b (longer ones set
 * FA_DEV_ERR_BOUND and are cut).  out: bf16 [N][Hq][D]; lse: optional float
 * [N][Hq].  The chunk's own k, v are read from k_ext / v_ext even if they
 * were stored first.  Hq / Hkv must divide 128 (query heads of a KV head are
 * packed into 128-row tensor-core tiles); other cases return
 * FA_ERR_UNSUPPORTED.  Every slab format is served. */
FA_API fa_status fa_paged_extend_attn(fa_cache* cache, int32_t layer, const void* q, const void* k_ext,
                               const void* v_ext, const int32_t* qo_indptr,
                               const int32_t* prefix_lens, const int32_t* block_table,
                               int32_t max_pages_per_seq, int32_t B, int32_t num_tokens,
                               int32_t max_q_len, int32_t max_prefix_len, void* out, float* lse,
                               void* stream);

/* Decode of n_b >= 1 new tokens per sequence whose k, v rows are already
 * stored: the verification step of speculative decoding, whose drafted
 * tokens attend over the target's paged cache ("FreeToken PR #898",
 * description: the assistant draft of speculative decoding reads the
 * target's slabs).
 * Query i of sequence b sits at position seq_lens[b] - n_b + i and attends
 * to keys [lo, its position] of the layer's regime (causal; sliding adds
 * q_pos - kv_pos < W), every key read from the slab through the block table.
 * The extend kernel computes it, with the chunk's keys taken from the slab.
 * q: bf16 [num_tokens][Hq][D], qo_indptr: int32 [B + 1] (device; n_b =
 * qo_indptr[b+1] - qo_indptr[b] <= max_q_len), seq_lens: int32 [B] (device;
 * lengths including the new tokens, <= max_seq_len; a length below n_b sets
 * FA_DEV_ERR_BOUND), block_table: int32 [B][max_pages_per_seq].  out: bf16
 * [num_tokens][Hq][D]; lse: optional float [num_tokens][Hq].  Every slab
 * format (8-bit codes and scales applied as in extend); Hq / Hkv must divide 128. */
FA_API fa_status fa_paged_decode_multi_attn(fa_cache* cache, int32_t layer, const void* q, const int32_t* qo_indptr,
                                            const int32_t* seq_lens, const int32_t* block_table,
                                            int32_t max_pages_per_seq, int32_t B, int32_t num_tokens,
                                            int32_t max_q_len, int32_t max_seq_len, void* out, float* lse,
                                            void* stream);

/* Synchronise `stream`, then read and clear the device error word of
 * `cache` on the current device (FA_DEV_ERR_* bits of every kernel launched
 * by calls on this cache since the last read; 0 = no error). */
FA_API fa_status fa_get_device_error(fa_cache* cache, int32_t* code, void* stream);

/* Message of the last failed call on this thread ("" if none). */
FA_API const char* fa_last_error(void);

/* Name of a status code. */
FA_API const char* fa_status_string(int32_t status);

/* Library ABI version (major * 100 + minor). */
FA_API int32_t fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
