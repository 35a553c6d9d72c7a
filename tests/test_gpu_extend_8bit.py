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
    reads every key from the slab)."""

    def __init__(self, layers, prefix, chunk, kv_dtype, seed, page_size=16, store_chunk=False):
        import full_attention_gb300 as fa
        self.fa, self.layers, self.kv, self.ps = fa, layers, kv_dtype, page_size
        self.prefix = np.asarray(prefix, np.int32)
        self.chunk = np.asarray(chunk, np.int32)
        self.B = len(prefix)
        total = self.prefix + self.chunk
        plan = W.plan_pages(np.maximum(total, 1), page_size, seed)
        self.bt_np = plan.block_table
        self.cache = fa.Cache(layers, plan.num_pages, page_size, kv_dtype)
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
            self.kx[o] = W.randn_bf16((max(self.N, 1), H, D), seed * 100 + 21 + 3 * o, dev)
            self.vx[o] = W.randn_bf16((max(self.N, 1), H, D), seed * 100 + 22 + 3 * o, dev)
            npre = int(self.prefix.sum())
            kp = W.randn_bf16((max(npre, 1), H, D), seed * 100 + 40 + 2 * o, dev)[:npre]
            vp = W.randn_bf16((max(npre, 1), H, D), seed * 100 + 41 + 2 * o, dev)[:npre]
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

    def oracle_extend(self, i):
        o = self.src[i]
        return oracle.paged_extend(self.layers, i, {o: self.oslabs[o]}, bits(self.q[i][: self.N]),
                                   bits(self.kx[o][: self.N]), bits(self.vx[o][: self.N]), self.indptr, self.prefix,
                                   self.bt_np, self.ps)

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
