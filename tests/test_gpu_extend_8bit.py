"""Extend and multi-token decode over the 8-bit per-token-head formats,
against the oracle.

The slab rows are seeded bf16 rows stored through the library (quantised on
the way); the oracle quantises the same rows with its own store and
dequantises them as code * scale in float64.  Chunk rows (extend) stay bf16.
Every slot the store does not write holds junk codes (e4m3: the NaN codes)
and NaN scales, which no visible key may read.  Tolerance as for extend:
max-abs 1e-2, relative L2 2e-2; lse within 2e-3 relative.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from paged_case import assert_close, bits

pytestmark = pytest.mark.gpu

FORMATS = [W.KV_INT8, W.KV_FP8]
IDS = ["int8", "fp8"]


def lay(kind, D, hq, hkv, Wn=0, src=W.KV_OWN):
    return W.layer(kind, D, hq, hkv, Wn, src)


class Case8:
    """Sequences with prefix_b stored tokens and chunk_b new ones.  With
    `store_chunk` the new tokens' rows are stored too (multi-token decode
    reads every key from the slab).  `mag` scales every k, v row (prefix and
    chunk) before it is rounded to bf16; `poke(kp, vp)` may edit the prefix
    rows before they are stored."""

    def __init__(self, layers, prefix, chunk, kv_dtype, seed, page_size=16, store_chunk=False, mag=1.0,
                 poke=None, split=None):
        import full_attention_gb300 as fa
        self.fa, self.layers, self.kv, self.ps = fa, layers, kv_dtype, page_size
        self.prefix = np.asarray(prefix, np.int32)
        self.chunk = np.asarray(chunk, np.int32)
        self.B = len(prefix)
        total = self.prefix + self.chunk
        plan = W.plan_pages(np.maximum(total, 1), page_size, seed)
        self.bt_np = plan.block_table
        self.cache = fa.Cache(layers, plan.num_pages, page_size, kv_dtype)
        if split is not None:
            # "tail": split as the bench launches do; "all": every job the workspace holds
            if split == "all":
                self.cache.set_flags(fa.FLAG_EXTEND_SPLIT_ALL)
            self.ws = fa.workspace(fa.extend_workspace_bytes(), "cuda")
            self.cache.bind_extend_workspace(self.ws)
        self.src = [self.cache.source(i) for i in range(len(layers))]
        self.slabs = self.cache.allocate("cuda")
        self.indptr = np.concatenate([[0], np.cumsum(self.chunk)]).astype(np.int32)
        self.N = int(self.indptr[-1])
        dev = "cuda"
        self.q, self.kx, self.vx, self.oslabs = {}, {}, {}, {}
        for i, d in enumerate(layers):
            self.q[i] = W.randn_bf16((max(self.N, 1), d["num_q_heads"], d["head_dim"]), seed * 100 + 20 + 3 * i, dev)
        store_q = oracle.store_fp8 if kv_dtype == W.KV_FP8 else oracle.store_int8
        code_t = np.uint8 if kv_dtype == W.KV_FP8 else np.int8
        for o, (k_s, v_s, ks_s, vs_s) in self.slabs.items():
            d = layers[o]
            H, D = d["num_kv_heads"], d["head_dim"]
            k_s.fill_(0x7F if kv_dtype == W.KV_FP8 else 77)
            v_s.fill_(0xFF if kv_dtype == W.KV_FP8 else -77)
            ks_s.fill_(float("nan"))
            vs_s.fill_(float("nan"))
            def gen(shape, sd):
                x = W.randn_bf16(shape, sd, dev)
                return x if mag == 1.0 else (x.float() * mag).to(torch.bfloat16)
            self.kx[o] = gen((max(self.N, 1), H, D), seed * 100 + 21 + 3 * o)
            self.vx[o] = gen((max(self.N, 1), H, D), seed * 100 + 22 + 3 * o)
            npre = int(self.prefix.sum())
            kp = gen((max(npre, 1), H, D), seed * 100 + 40 + 2 * o)[:npre]
            vp = gen((max(npre, 1), H, D), seed * 100 + 41 + 2 * o)[:npre]
            if poke is not None:
                poke(kp, vp)
            slots = [W.slots_for_positions(self.bt_np[b], np.arange(0, int(self.prefix[b])), page_size)
                     for b in range(self.B)]
            slots = np.concatenate(slots).astype(np.int32)
            rows_k, rows_v, all_slots = [kp], [vp], [slots]
            if store_chunk and self.N:
                cs = np.concatenate([W.slots_for_positions(self.bt_np[b], np.arange(int(self.prefix[b]),
                                                                                     int(total[b])), page_size)
                                     for b in range(self.B)]).astype(np.int32)
                rows_k.append(self.kx[o][: self.N])
                rows_v.append(self.vx[o][: self.N])
                all_slots.append(cs)
            kr, vr = torch.cat(rows_k), torch.cat(rows_v)
            sl = np.concatenate(all_slots).astype(np.int32)
            if sl.size:
                self.cache.store(o, kr, vr, torch.from_numpy(sl).cuda())
            ck = np.zeros((plan.num_pages, H, page_size, D), code_t)
            cv = np.zeros_like(ck)
            sk = np.zeros((plan.num_pages, H, page_size), np.float32)
            sv = np.zeros_like(sk)
            if sl.size:
                store_q(ck, cv, sk, sv, bits(kr), bits(vr), sl, page_size)
            self.oslabs[o] = (ck, cv, sk, sv)
        self.bt = torch.from_numpy(self.bt_np).cuda()
        self.indptr_dev = torch.from_numpy(self.indptr).cuda()
        self.prefix_dev = torch.from_numpy(self.prefix).cuda()
        self.lens_dev = torch.from_numpy(total.astype(np.int32)).cuda()
        torch.cuda.synchronize()

    def _out(self, i):
        d = self.layers[i]
        out = torch.full((max(self.N, 1), d["num_q_heads"], d["head_dim"]), float("nan"), dtype=torch.bfloat16,
                         device="cuda")
        lse = torch.full((max(self.N, 1), d["num_q_heads"]), float("nan"), dtype=torch.float32, device="cuda")
        return out, lse

    def extend(self, i):
        o = self.src[i]
        out, lse = self._out(i)
        self.cache.extend(i, self.q[i][: self.N], self.kx[o][: self.N], self.vx[o][: self.N], self.indptr_dev,
                          self.prefix_dev, self.bt, int(self.chunk.max()), int(max(self.prefix.max(), 0)), out, lse)
        return out[: self.N], lse[: self.N]

    def oracle_extend(self, i, rows=None):
        o = self.src[i]
        return oracle.paged_extend(self.layers, i, {o: self.oslabs[o]}, bits(self.q[i][: self.N]),
                                   bits(self.kx[o][: self.N]), bits(self.vx[o][: self.N]), self.indptr, self.prefix,
                                   self.bt_np, self.ps, rows=rows)

    def decode_multi(self, i):
        out, lse = self._out(i)
        total = self.prefix + self.chunk
        self.cache.decode_multi(i, self.q[i][: self.N], self.indptr_dev, self.lens_dev, self.bt,
                                int(self.chunk.max()), int(total.max()), out, lse)
        return out[: self.N], lse[: self.N]

    def oracle_decode_multi(self, i):
        """New token j of sequence b is a decode query at position P_b + j:
        one virtual decode sequence of length P_b + j + 1 per new token."""
        o = self.src[i]
        bt = np.stack([self.bt_np[b] for b in range(self.B) for _ in range(int(self.chunk[b]))])
        lens = np.array([int(self.prefix[b]) + j + 1 for b in range(self.B) for j in range(int(self.chunk[b]))],
                        np.int32)
        return oracle.paged_decode(self.layers, i, {o: self.oslabs[o]}, bits(self.q[i][: self.N]), bt, lens,
                                   self.ps)


def _check(got, ref, what):
    out, lse = got
    ref_out, ref_lse = ref
    assert_close(out, ref_out, what=what)
    g = lse.double().cpu().numpy()
    assert np.all(np.abs(g - ref_lse) <= 2e-3 * np.maximum(1.0, np.abs(ref_lse))), f"{what}: lse"


EXTEND = [
    # (layer, prefix, chunk)
    (lay(W.SLIDING, 256, 4, 2, 48), [40, 0, 100, 17], [37, 20, 130, 1]),
    (lay(W.FULL, 512, 8, 1), [40, 0, 100, 17], [37, 20, 130, 1]),
    (lay(W.FULL, 256, 16, 8), [64, 3], [64, 200]),
    (lay(W.SLIDING, 512, 16, 2, 100), [300, 33], [90, 160]),
]


@pytest.mark.parametrize("kv_dtype", FORMATS, ids=IDS)
@pytest.mark.parametrize("spec", EXTEND, ids=[f"{'F' if s[0]['kind'] == 0 else 'S'}{s[0]['head_dim']}"
                                              f"_g{s[0]['num_q_heads'] // s[0]['num_kv_heads']}_W{s[0]['window']}"
                                              for s in EXTEND])
def test_8bit_extend(spec, kv_dtype):
    layer, prefix, chunk = spec
    c = Case8([layer], prefix, chunk, kv_dtype, seed=31)
    _check(c.extend(0), c.oracle_extend(0), "8-bit extend")
    assert c.fa.device_error() == 0


@pytest.mark.parametrize("kv_dtype", FORMATS, ids=IDS)
@pytest.mark.parametrize("spec", EXTEND, ids=[f"{'F' if s[0]['kind'] == 0 else 'S'}{s[0]['head_dim']}"
                                              f"_g{s[0]['num_q_heads'] // s[0]['num_kv_heads']}_W{s[0]['window']}"
                                              for s in EXTEND])
def test_8bit_extend_split(spec, kv_dtype):
    """Every job split over two CTAs and merged through the workspace (the
    8-bit exponent base, 2^7 below the running maximum, joins the merge)."""
    layer, prefix, chunk = spec
    c = Case8([layer], prefix, chunk, kv_dtype, seed=31, split="all")
    _check(c.extend(0), c.oracle_extend(0), "8-bit split extend")
    assert c.fa.device_error() == 0


@pytest.mark.parametrize("kv_dtype", FORMATS, ids=IDS)
def test_8bit_extend_shared_layer(kv_dtype):
    layers = [lay(W.SLIDING, 256, 8, 2, 64), lay(W.FULL, 512, 8, 1), lay(W.SLIDING, 256, 8, 2, 64, W.KV_AUTO)]
    c = Case8(layers, [50, 130], [70, 20], kv_dtype, seed=32)
    assert c.src == [0, 1, 0]
    for i in range(3):
        _check(c.extend(i), c.oracle_extend(i), f"8-bit extend layer {i}")
    assert c.fa.device_error() == 0


MULTI = [
    (lay(W.FULL, 512, 8, 1), [40, 0, 100, 17], [4, 1, 8, 3]),
    (lay(W.SLIDING, 256, 8, 1, 64), [40, 5, 100, 300], [4, 1, 8, 5]),
    (lay(W.SLIDING, 256, 16, 8, 1024), [2000, 64], [7, 16]),
]


@pytest.mark.parametrize("kv_dtype", FORMATS, ids=IDS)
@pytest.mark.parametrize("spec", MULTI, ids=[f"{'F' if s[0]['kind'] == 0 else 'S'}{s[0]['head_dim']}"
                                             f"_g{s[0]['num_q_heads'] // s[0]['num_kv_heads']}_W{s[0]['window']}"
                                             for s in MULTI])
def test_8bit_multi_token_decode(spec, kv_dtype):
    layer, prefix, new = spec
    c = Case8([layer], prefix, new, kv_dtype, seed=33, store_chunk=True)
    _check(c.decode_multi(0), c.oracle_decode_multi(0), "8-bit multi-token decode")
    assert c.fa.device_error() == 0


EDGE = [
    # (layer, prefix, chunk, page size)
    (lay(W.SLIDING, 256, 8, 1, 1), [20, 0], [45, 16], 16),          # W = 1: only the current token
    (lay(W.FULL, 256, 2, 2), [0, 129], [257, 1], 16),               # empty prefix; a single new token
    (lay(W.SLIDING, 512, 8, 2, 40), [95, 33, 64], [33, 96, 1], 32), # page size 32
]


@pytest.mark.parametrize("kv_dtype", FORMATS, ids=IDS)
@pytest.mark.parametrize("spec", EDGE, ids=["W1", "empty_prefix", "page32"])
def test_8bit_extend_edges(spec, kv_dtype):
    layer, prefix, chunk, ps = spec
    c = Case8([layer], prefix, chunk, kv_dtype, seed=34, page_size=ps)
    _check(c.extend(0), c.oracle_extend(0), "8-bit extend edge")
    assert c.fa.device_error() == 0


@pytest.mark.parametrize("kv_dtype", FORMATS, ids=IDS)
def test_8bit_chunked_prefill_workload(kv_dtype):
    """The chunked-prefill workload (4 prompts of 4096 tokens in 512-token
    chunks, sliding D 256 W 1024 with 16 q / 8 KV heads and full D 512 with
    16 q / 2 KV heads) over 8-bit slabs, at full size: chunks 0, 3 and 7 of
    both layers, on sampled rows that include the first and last rows and the
    boundary between the first two sequences, every query head of each.  The
    split workspace is bound as in the bench."""
    w = W.chunked_prefill()
    B, Cn = w.batch, w.chunk
    rng = np.random.default_rng(5)
    for ci in (0, 3, 7):
        P = ci * Cn
        c = Case8(w.layers, [P] * B, [Cn] * B, kv_dtype, seed=40 + ci, split="tail")
        for li in range(len(w.layers)):
            out, lse = c.extend(li)
            d = w.layers[li]
            toks = sorted(set(rng.choice(c.N, size=16, replace=False).tolist() + [0, c.N - 1, Cn - 1, Cn]))
            rows = [(t, j) for t in toks for j in range(d["num_q_heads"])]
            ref_out, ref_lse = c.oracle_extend(li, rows=rows)
            idx = torch.tensor(toks)
            _check((out[idx], lse[idx]), (ref_out[toks], ref_lse[toks]), f"{IDS[FORMATS.index(kv_dtype)]} chunk {ci} layer {li}")
        assert c.fa.device_error() == 0


@pytest.mark.parametrize("kv_dtype", FORMATS, ids=IDS)
@pytest.mark.parametrize("mag", [1e-3, 1e-4], ids=["1e-3", "1e-4"])
def test_8bit_extend_small_magnitudes(mag, kv_dtype):
    """Rows of small magnitude: the prefix codes enter the MMAs exactly and
    their scales multiply in fp32, so only the chunk rows (bf16 as f16, some
    elements f16 subnormals) and the f16 weights round; the relative L2 error
    stays within the float tolerance."""
    for layer in (lay(W.SLIDING, 256, 8, 2, 64), lay(W.FULL, 512, 8, 1)):
        c = Case8([layer], [70, 150], [90, 33], kv_dtype, seed=35, mag=mag)
        _check(c.extend(0), c.oracle_extend(0), f"small rows x{mag}")
        assert c.fa.device_error() == 0


BIG_IN, BIG_OUT = 65280.0, 65536.0   # the bf16 values on either side of f16's largest (65504)


@pytest.mark.parametrize("kv_dtype", FORMATS, ids=IDS)
def test_8bit_extend_f16_range_inside(kv_dtype):
    """Values of 65280, just inside the f16 range, set no error bit.  With
    them in a chunk key row and a stored prefix key row the result also
    matches the oracle: those keys win or lose their softmax rows by
    thousands, a well-conditioned case.  A q element that large is not
    compared: its scores against the other keys are about 4000 times the
    key values, so a rounding of one part in 2^12 in the f16 chunk keys
    moves them by several units and the softmax weights with them, on any
    f16 path.  q, V and the prefix V rows are checked for the error bit."""
    def poke_k(kp, vp):
        kp[3, 0, 5] = -BIG_IN
    c = Case8([lay(W.FULL, 256, 4, 1)], [40, 20], [30, 10], kv_dtype, seed=36, poke=poke_k)
    c.kx[0][2, 0, 0] = BIG_IN
    _check(c.extend(0), c.oracle_extend(0), "key values at 65280")
    assert c.fa.device_error() == 0

    def poke_v(kp, vp):
        vp[7, 0, 9] = BIG_IN
    c = Case8([lay(W.FULL, 256, 4, 1)], [40, 20], [30, 10], kv_dtype, seed=36, poke=poke_v)
    c.q[0][4, 1, 11] = BIG_IN
    c.vx[0][5, 0, 7] = -BIG_IN
    c.extend(0)
    assert c.fa.device_error() == 0


@pytest.mark.parametrize("kv_dtype", FORMATS, ids=IDS)
@pytest.mark.parametrize("where", ["q", "k_ext", "v_ext"])
def test_8bit_extend_f16_range_outside_sets_error_bit(where, kv_dtype):
    """A value of 65536, just past the f16 range, in q or in a chunk row
    (the values the kernel converts to f16): it saturates and sets
    FA_DEV_ERR_RANGE."""
    c = Case8([lay(W.FULL, 256, 4, 1)], [40, 20], [30, 10], kv_dtype, seed=37)
    if where == "q":
        c.q[0][4, 1, 11] = BIG_OUT
    if where == "k_ext":
        c.kx[0][2, 0, 0] = -BIG_OUT
    if where == "v_ext":
        c.vx[0][5, 0, 7] = BIG_OUT
    c.extend(0)
    assert c.fa.device_error() == c.fa.DEV_ERR_RANGE


@pytest.mark.parametrize("kv_dtype", FORMATS, ids=IDS)
@pytest.mark.parametrize("where", ["prefix_k", "prefix_v"])
def test_8bit_extend_large_prefix_rows(where, kv_dtype):
    """Stored prefix rows have no f16 limit: their codes enter the MMAs as
    exact f16 values and their scales apply in fp32 (K to the scores, V to
    the weights).  A key element of 65536 keeps parity with the oracle (the
    key wins or loses its rows by thousands); V elements of -65536 and 3e7
    (a V scale past f16's range in both formats) match it to the output's
    bf16 precision, relative to the largest output.  No error bit is set."""
    def poke(kp, vp):
        if where == "prefix_k":
            kp[3, 0, 5] = BIG_OUT
        else:
            vp[7, 0, 9] = -BIG_OUT
            vp[21, 0, 30] = 3.0e7
    for layer in (lay(W.FULL, 256, 4, 1), lay(W.SLIDING, 512, 8, 2, 40)):
        c = Case8([layer], [40, 20], [30, 10], kv_dtype, seed=37, poke=poke)
        out, lse = c.extend(0)
        ref_out, ref_lse = c.oracle_extend(0)
        scale = max(1.0, float(np.abs(ref_out).max()))
        assert_close(out, ref_out, atol=1e-2 * scale, what=f"{where} large")
        g = lse.double().cpu().numpy()
        assert np.all(np.abs(g - ref_lse) <= 2e-3 * np.maximum(1.0, np.abs(ref_lse))), f"{where}: lse"
        assert c.fa.device_error() == 0


@pytest.mark.parametrize("kv_dtype", FORMATS, ids=IDS)
def test_8bit_decode_f16_range(kv_dtype):
    """8-bit decode converts q to f16: 65280 passes without an error bit,
    65536 saturates and sets FA_DEV_ERR_RANGE."""
    c = Case8([lay(W.FULL, 512, 8, 1)], [40, 90], [1, 1], kv_dtype, seed=38, store_chunk=True)
    max_len = int(c.lens_dev.max())
    ws = c.fa.workspace(c.cache.decode_workspace_bytes(0, c.B, max_len))
    for val, want in ((BIG_IN, 0), (BIG_OUT, c.fa.DEV_ERR_RANGE)):
        q = c.q[0][: c.N].clone()
        q[1, 3, 100] = val
        out = torch.empty_like(q)
        c.cache.decode(0, q, c.bt, c.lens_dev, max_len, out, None, ws)
        assert c.fa.device_error() == want
