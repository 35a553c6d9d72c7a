"""fp64 CPU oracle for Gemma-4-style paged-KV attention.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, links or runs
this package: only the tests, the smoke check and the CPU baseline of the
benchmark do.  It shares no code with the CUDA library (no kernels, headers,
helpers, tables or constants); both sides only take their inputs from the
seeded generators in ``workloads.py``.

It computes the plain definitions, slowly and obviously:

* layer map -- which slab a layer reads, and what a token costs in bytes;
* the paged KV store (a bf16 copy, or int8 or fp8 e4m3 per-token-head codes
  with an fp32 scale), computed in fp32 where bit-exactness with the GPU is
  required;
* decode and extend attention over the *logically gathered* KV in float64:
  gather the visible rows through the block table, then softmax(scale q.K) V.

Conventions (the same ones the C boundary documents):

* bf16 values travel as numpy ``uint16`` bit patterns; int8 codes as ``int8``;
  fp8 e4m3 codes as ``uint8`` bit patterns.
* slab layout ``[num_pages][Hkv][page_size][D]``; scales ``[num_pages][Hkv][page_size]``.
* a slot is ``page * page_size + offset``; a negative slot is skipped.
* query head ``j`` reads KV head ``j // (Hq / Hkv)`` (contiguous groups).
* full layers: keys ``k <= q``; sliding layers: ``k <= q`` and ``q - k < W``
  (W counts the current token, so W = 1024 sees 1023 earlier positions).

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
against something other than itself (a library attention routine on dense
inputs, closed forms, invariants, or numbers the pages print).
"""
from __future__ import annotations

import numpy as np

FULL = 0
SLIDING = 1
KV_OWN = -1
KV_AUTO = -2
KV_BF16 = 0
KV_INT8 = 1
KV_FP8 = 2


# ---------------------------------------------------------------------------
# bf16 bit patterns
# ---------------------------------------------------------------------------

def bf16_to_f32(bits) -> np.ndarray:
    """bf16 bit patterns -> float32 (exact: bf16 is the top half of an fp32)."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32)


def bf16_to_f64(bits) -> np.ndarray:
    return bf16_to_f32(bits).astype(np.float64)


# ---------------------------------------------------------------------------
# layer map
# ---------------------------------------------------------------------------

class UnsupportedLayout(ValueError):
    """A layer layout the method refuses (e.g. a KV-shared layer with no source)."""


def resolve_kv_sources(layers) -> list:
    """Slab owner of every layer: -1 if the layer owns a slab, else its source.

    "FreeToken PR #898: read the source layer's kv slab on kv-shared layers",
    description, first bullet: a KV-shared layer reads the slab of the last
    earlier layer of its attention type; a shared layer with no such earlier
    layer is refused (review thread: NotImplementedError).  A source that is
    itself shared is not a slab owner, so it does not qualify.  An explicit
    source must be an earlier owning layer of the same kind with the same KV
    geometry (head_dim, num_kv_heads), because the shared layer reads its slab
    as is.
    """
    src = []
    for i, L in enumerate(layers):
        want = L["kv_source"]
        if want == KV_OWN:
            src.append(-1)
            continue
        owners = [j for j in range(i) if src[j] == -1 and layers[j]["kind"] == L["kind"]]
        if not owners:
            raise UnsupportedLayout(f"layer {i}: KV-shared layer with no earlier layer of its kind")
        s = owners[-1] if want == KV_AUTO else want
        if s not in owners:
            raise UnsupportedLayout(f"layer {i}: source {s} is not an earlier owning layer of its kind")
        o = layers[s]
        if o["head_dim"] != L["head_dim"] or o["num_kv_heads"] != L["num_kv_heads"]:
            raise UnsupportedLayout(f"layer {i}: KV geometry differs from source {s}")
        src.append(s)
    return src


def slab_owner(layers, li: int) -> int:
    s = resolve_kv_sources(layers)[li]
    return li if s == -1 else s


def slab_counts(layers) -> dict:
    """Number of slabs per attention kind: one per owning layer."""
    src = resolve_kv_sources(layers)
    out = {FULL: 0, SLIDING: 0}
    for L, s in zip(layers, src):
        if s == -1:
            out[L["kind"]] += 1
    return out


def kv_bytes_per_token(layers, kind: int, kv_dtype: int) -> int:
    """Bytes one token occupies across the slabs of the owning layers of `kind`.

    Per owning layer and KV head: K and V rows of head_dim elements (2 bytes in
    bf16, 1 byte in the 8-bit formats) plus, in the int8 and fp8 per-token-head
    formats, one fp32 scale each for K and V.  Shared layers cost nothing.  ("FreeToken PR #898",
    description bullets on kv_cache_group_specs and the per-token-head formats;
    the "End to end" section prints the resulting unit_bytes.)
    """
    src = resolve_kv_sources(layers)
    total = 0
    for L, s in zip(layers, src):
        if L["kind"] != kind or s != -1:
            continue
        if kv_dtype == KV_BF16:
            per_row = 2 * L["head_dim"]
        else:
            per_row = L["head_dim"] + 4
        total += 2 * L["num_kv_heads"] * per_row
    return total


# ---------------------------------------------------------------------------
# paged KV store
# ---------------------------------------------------------------------------

def store_bf16(slab_k, slab_v, k, v, slot_mapping, page_size: int) -> None:
    """Write token t's post-RoPE rows k[t], v[t] ([Hkv][D] bf16 bits) into
    slot slot_mapping[t] = page * page_size + offset of the slab, in place.
    Negative slots are padding and are skipped.  ("unsloth commit dee9371":
    the store layer writes its post-rotary k, v into its PagedKVCache.)"""
    for t, slot in enumerate(np.asarray(slot_mapping)):
        slot = int(slot)
        if slot < 0:
            continue
        page, off = divmod(slot, page_size)
        slab_k[page, :, off, :] = k[t]
        slab_v[page, :, off, :] = v[t]


def quantize_int8_per_token_head(x_bits):
    """int8 per-token-head quantisation of rows x[..., D] (bf16 bits).

    For each row, in fp32 with IEEE round-to-nearest-even: a = max |x_d|,
    s = a / 127, c_d = clamp(rint(x_d / s), -127, 127), with rint rounding
    half to even; an all-zero row gets s = 0 and codes 0.  Returns
    (codes int8 [..., D], scale float32 [...]).  ("FreeToken PR #898": the
    int8_per_token_head format keeps int8 codes plus an fp32 scale per
    token and KV head, separately for K and V.)
    """
    x = bf16_to_f32(x_bits)
    a = np.max(np.abs(x), axis=-1).astype(np.float32)
    s = (a / np.float32(127.0)).astype(np.float32)
    zero = a == np.float32(0.0)
    s_div = np.where(zero, np.float32(1.0), s).astype(np.float32)
    q = (x / s_div[..., None]).astype(np.float32)
    c = np.clip(np.rint(q), -127.0, 127.0)
    c = np.where(zero[..., None], 0.0, c)
    return c.astype(np.int8), s


# fp8 e4m3 ("FreeToken PR #898", description: the fp8_per_token_head format,
# stored and looked up like the int8 one).  The pages name the format only; the
# encoding is E4M3 of the OCP 8-bit floating point specification, the variant
# without infinities, whose largest finite magnitude is 448.

E4M3_MAX = 448.0


def e4m3_value(codes) -> np.ndarray:
    """float64 value of e4m3 bit patterns (uint8).

    Bit 7 is the sign, bits 6..3 an exponent field e with bias 7, bits 2..0 a
    mantissa m.  e > 0 gives (1 + m/8) * 2**(e - 7); e = 0 gives the subnormal
    (m/8) * 2**-6.  The patterns 0x7F and 0xFF are NaN; there are no
    infinities, so 0x7E = 448 is the largest finite magnitude.
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    e = (c >> 3) & 0xF
    m = (c & 7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2((e - 7).astype(np.float64)))
    mag = np.where((c & 0x7F) == 0x7F, np.nan, mag)
    return np.where((c & 0x80) != 0, -mag, mag)


def e4m3_round(y) -> np.ndarray:
    """e4m3 codes of float32 values y: the nearest finite e4m3 value, a tie
    going to the code with the even mantissa, magnitudes above 448
    saturating to 448.  The sign is kept, so a negative value that rounds to
    zero gives 0x80.  (Round-to-nearest-even with saturation to the finite
    range: the plain reading for a quantised cache, which must never hold NaN.)"""
    y = np.asarray(y, dtype=np.float32)
    mags = e4m3_value(np.arange(0x7F, dtype=np.uint8))   # codes 0 .. 126, ascending
    a = np.abs(y).astype(np.float64)
    lo = np.clip(np.searchsorted(mags, a, side="right") - 1, 0, 126)   # mags[lo] <= a
    hi = np.minimum(lo + 1, 126)
    d_lo = a - mags[lo]
    d_hi = mags[hi] - a
    up = (hi > lo) & ((d_hi < d_lo) | ((d_hi == d_lo) & (lo % 2 == 1)))
    code = np.where(up, hi, lo).astype(np.uint8)
    return np.where(np.signbit(y), code | np.uint8(0x80), code).astype(np.uint8)


def quantize_fp8_per_token_head(x_bits):
    """fp8 e4m3 per-token-head quantisation of rows x[..., D] (bf16 bits).

    For each row, in fp32 with IEEE round-to-nearest-even: a = max |x_d|,
    s = a / 448, c_d = e4m3_round(x_d / s); an all-zero row gets s = 0 and
    codes 0.  Returns (codes uint8 [..., D], scale float32 [...]).  The scale
    maps the row's largest magnitude onto the largest finite e4m3 value, as
    the int8 format maps it onto 127.
    """
    x = bf16_to_f32(x_bits)
    a = np.max(np.abs(x), axis=-1).astype(np.float32)
    s = (a / np.float32(E4M3_MAX)).astype(np.float32)
    zero = a == np.float32(0.0)
    s_div = np.where(zero, np.float32(1.0), s).astype(np.float32)
    q = (x / s_div[..., None]).astype(np.float32)
    c = np.where(zero[..., None], np.uint8(0), e4m3_round(q))
    return c.astype(np.uint8), s


def _store_quantised(quantize, codes_k, codes_v, scale_k, scale_v, k, v, slot_mapping, page_size: int) -> None:
    ck, sk = quantize(k)
    cv, sv = quantize(v)
    for t, slot in enumerate(np.asarray(slot_mapping)):
        slot = int(slot)
        if slot < 0:
            continue
        page, off = divmod(slot, page_size)
        codes_k[page, :, off, :] = ck[t]
        codes_v[page, :, off, :] = cv[t]
        scale_k[page, :, off] = sk[t]
        scale_v[page, :, off] = sv[t]


def store_int8(codes_k, codes_v, scale_k, scale_v, k, v, slot_mapping, page_size: int) -> None:
    """Quantise and write rows like store_bf16, into int8 code slabs
    [num_pages][Hkv][ps][D] and fp32 scale arrays [num_pages][Hkv][ps]."""
    _store_quantised(quantize_int8_per_token_head, codes_k, codes_v, scale_k, scale_v, k, v, slot_mapping,
                     page_size)


def store_fp8(codes_k, codes_v, scale_k, scale_v, k, v, slot_mapping, page_size: int) -> None:
    """Quantise and write rows like store_bf16, into e4m3 code slabs (uint8)
    [num_pages][Hkv][ps][D] and fp32 scale arrays [num_pages][Hkv][ps]."""
    _store_quantised(quantize_fp8_per_token_head, codes_k, codes_v, scale_k, scale_v, k, v, slot_mapping,
                     page_size)


# ---------------------------------------------------------------------------
# attention over the logically gathered KV
# ---------------------------------------------------------------------------

def visible_keys(q_pos: int, kind: int, window: int) -> tuple:
    """Inclusive key range [lo, q_pos] a query at q_pos attends to.

    Full layers are purely causal; sliding layers are causal and
    q_pos - kv_pos < W ("unsloth gemma4_flex_inference.py history", commit
    "block mask per attention regime"; "pegainfer issue #807", Description:
    Gemma counts the current token inside its window).
    """
    if kind == FULL:
        return 0, q_pos
    return max(0, q_pos - window + 1), q_pos


def gather_rows(slab, scales, block_table_row, positions, h: int, page_size: int) -> np.ndarray:
    """Logical rows at `positions` of KV head h, as float64 [n][D]: page =
    block_table_row[pos // page_size], offset = pos % page_size.  bf16 slabs
    (uint16) are widened exactly; int8 slabs (int8) and fp8 slabs (uint8 e4m3
    bit patterns) are dequantised as value(code) * scale."""
    positions = np.asarray(positions, dtype=np.int64)
    pages = np.asarray(block_table_row, dtype=np.int64)[positions // page_size]
    if np.any(pages < 0):
        raise IndexError("visible position maps to an unassigned page")
    offs = positions % page_size
    rows = slab[pages, h, offs, :]
    if slab.dtype == np.uint16:
        return bf16_to_f64(rows)
    sc = scales[pages, h, offs].astype(np.float64)
    vals = e4m3_value(rows) if slab.dtype == np.uint8 else rows.astype(np.float64)
    return vals * sc[:, None]


def softmax_attention(q, K, V, sm_scale: float):
    """out = softmax(sm_scale * K q) V for one query row, in float64.
    Returns (out [D], lse = log sum exp of the scaled scores, p [n])."""
    s = float(sm_scale) * (K @ q)
    m = np.max(s)
    e = np.exp(s - m)
    l = np.sum(e)
    p = e / l
    return p @ V, m + np.log(l), p


def _owner_arrays(slabs, owner):
    entry = slabs[owner]
    k, v = entry[0], entry[1]
    ks = entry[2] if len(entry) > 2 else None
    vs = entry[3] if len(entry) > 3 else None
    return k, v, ks, vs


def paged_decode(layers, li: int, slabs, q, block_table, seq_lens, page_size: int,
                 rows=None):
    """Decode attention of layer li for every (sequence, query head).

    q: bf16 bits [B][Hq][D]; block_table int32 [B][max_pages]; seq_lens [B]
    counts the current token, which is already stored, so q_pos = L - 1.
    A KV-shared layer reads its source's slab and scales ("FreeToken PR
    #898", description).  slabs: {owner layer: (k, v[, k_scale, v_scale])}.
    `rows`, if given, is a list of (b, j) pairs to compute (others stay 0).
    Returns (out float64 [B][Hq][D], lse float64 [B][Hq]); a sequence with
    L <= 0 has out 0 and lse -inf.
    """
    L = layers[li]
    owner = slab_owner(layers, li)
    ks, vs, kscale, vscale = _owner_arrays(slabs, owner)
    B, Hq, D = q.shape
    Hkv = L["num_kv_heads"]
    g = Hq // Hkv
    out = np.zeros((B, Hq, D), dtype=np.float64)
    lse = np.full((B, Hq), -np.inf, dtype=np.float64)
    want = None if rows is None else set((int(b), int(j)) for b, j in rows)
    for b in range(B):
        n = int(seq_lens[b])
        if n <= 0:
            continue
        lo, hi = visible_keys(n - 1, L["kind"], L["window"])
        pos = np.arange(lo, hi + 1)
        for h in range(Hkv):
            heads = [j for j in range(h * g, (h + 1) * g) if want is None or (b, j) in want]
            if not heads:
                continue
            K = gather_rows(ks, kscale, block_table[b], pos, h, page_size)
            V = gather_rows(vs, vscale, block_table[b], pos, h, page_size)
            for j in heads:
                o, s, _ = softmax_attention(bf16_to_f64(q[b, j]), K, V, L["sm_scale"])
                out[b, j] = o
                lse[b, j] = s
    return out, lse


def paged_extend(layers, li: int, slabs, q, k_ext, v_ext, qo_indptr, prefix_lens,
                 block_table, page_size: int, rows=None):
    """Extend (chunked prefill) attention of layer li.

    Sequence b contributes queries qo_indptr[b] .. qo_indptr[b+1]-1; query i
    sits at position P_b + i, P_b = prefix_lens[b].  Keys at positions < P_b
    come from the paged slab (through the block table, dequantised for int8);
    keys at P_b + j come from the current chunk k_ext / v_ext [N][Hkv][D]
    (bf16, never quantised).  For a shared layer the chunk is the source
    layer's current k, v ("FreeToken PR #898", description: the extend kernel
    takes the current chunk from k_extend / v_extend; "unsloth commit dee9371":
    shared layers read the store layer's post-rotary k, v on prefill).
    `rows`: optional list of (token index, q head) pairs to compute.
    Returns out float64 [N][Hq][D] and lse float64 [N][Hq].
    """
    L = layers[li]
    owner = slab_owner(layers, li)
    ks, vs, kscale, vscale = _owner_arrays(slabs, owner)
    N, Hq, D = q.shape
    Hkv = L["num_kv_heads"]
    g = Hq // Hkv
    out = np.zeros((N, Hq, D), dtype=np.float64)
    lse = np.full((N, Hq), -np.inf, dtype=np.float64)
    want = None if rows is None else set((int(t), int(j)) for t, j in rows)
    B = len(prefix_lens)
    for b in range(B):
        s0, s1 = int(qo_indptr[b]), int(qo_indptr[b + 1])
        n = s1 - s0
        P = int(prefix_lens[b])
        if n <= 0:
            continue
        first_lo, _ = visible_keys(P, L["kind"], L["window"])
        pref = np.arange(first_lo, P)
        for h in range(Hkv):
            Kp = gather_rows(ks, kscale, block_table[b], pref, h, page_size)
            Vp = gather_rows(vs, vscale, block_table[b], pref, h, page_size)
            Kc = bf16_to_f64(k_ext[s0:s1, h])
            Vc = bf16_to_f64(v_ext[s0:s1, h])
            Kall = np.concatenate([Kp, Kc], axis=0)   # positions first_lo .. P + n - 1
            Vall = np.concatenate([Vp, Vc], axis=0)
            for i in range(n):
                lo, hi = visible_keys(P + i, L["kind"], L["window"])
                a, z = lo - first_lo, hi - first_lo + 1
                for j in range(h * g, (h + 1) * g):
                    if want is not None and (s0 + i, j) not in want:
                        continue
                    o, s, _ = softmax_attention(bf16_to_f64(q[s0 + i, j]), Kall[a:z], Vall[a:z],
                                                L["sm_scale"])
                    out[s0 + i, j] = o
                    lse[s0 + i, j] = s
    return out, lse
