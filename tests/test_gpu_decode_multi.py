"""Multi-token decode (fa_paged_decode_multi_attn) against the oracle.

Each case pages a seeded context into a permuted pool, stores the n_b new
tokens' rows into their slots through the library, and decodes those n_b
queries with every key read from the slab.  The oracle is the extend
oracle with the new rows as the chunk (the same values the slab holds), so
query i of sequence b sits at position L_b - n_b + i.  Tolerance as for
extend: max-abs 1e-2, relative L2 2e-2; lse within 2e-3.
"""
import numpy as np
import pytest
import torch

import workloads as W
from paged_case import assert_close
from test_gpu_extend import ExtendCase

pytestmark = pytest.mark.gpu


def lay(kind, D, hq, hkv, Wn=0, src=W.KV_OWN):
    return W.layer(kind, D, hq, hkv, Wn, src)


def _store_chunk(c, i):
    """Store layer i's (its source's) chunk rows k_ext / v_ext at positions P .. P + n - 1."""
    o = c.src[i]
    slots = np.concatenate([W.slots_for_positions(c.bt_np[b], np.arange(int(c.prefix[b]),
                                                                        int(c.prefix[b] + c.chunk[b])), c.ps)
                            for b in range(c.B)]).astype(np.int32)
    c.cache.store(o, c.kx[o][: c.N], c.vx[o][: c.N], torch.from_numpy(slots).cuda())


def _decode_multi(c, i):
    d = c.layers[i]
    lens = torch.from_numpy((c.prefix + c.chunk).astype(np.int32)).cuda()
    out = torch.full((c.N, d["num_q_heads"], d["head_dim"]), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((c.N, d["num_q_heads"]), float("nan"), dtype=torch.float32, device="cuda")
    c.cache.decode_multi(i, c.q[i][: c.N], c.indptr_dev, lens, c.bt, int(c.chunk.max()), int(lens.max()), out, lse)
    return out, lse


CASES = [
    # (layer, context before the new tokens, new tokens per sequence)
    (lay(W.FULL, 512, 8, 1), [40, 0, 100, 17, 300], [4, 1, 8, 3, 5]),
    (lay(W.SLIDING, 256, 8, 1, 64), [40, 5, 100, 17, 300], [4, 1, 8, 3, 5]),
    (lay(W.SLIDING, 256, 16, 8, 1024), [2000, 64, 1500], [7, 16, 2]),
    (lay(W.FULL, 256, 16, 2), [64, 3], [64, 200]),
    (lay(W.SLIDING, 512, 16, 2, 100), [300, 33], [9, 160]),
    (lay(W.SLIDING, 256, 8, 1, 1), [20, 0], [3, 6]),
]


@pytest.mark.parametrize("spec", CASES, ids=[f"{'F' if s[0]['kind'] == 0 else 'S'}{s[0]['head_dim']}"
                                             f"_g{s[0]['num_q_heads'] // s[0]['num_kv_heads']}_W{s[0]['window']}"
                                             for s in CASES])
def test_multi_token_decode(spec):
    layer, prefix, new = spec
    c = ExtendCase([layer], prefix, new, seed=12, poison_tail=False)
    _store_chunk(c, 0)
    out, lse = _decode_multi(c, 0)
    ref = c.oracle(0)
    assert_close(out, ref, what="multi-token decode")
    g = lse.double().cpu().numpy()
    assert np.all(np.abs(g - c.oracle_lse) <= 2e-3 * np.maximum(1.0, np.abs(c.oracle_lse)))
    assert c.fa.device_error() == 0


@pytest.mark.parametrize("spec", CASES[:3], ids=["F512_g8", "S256_g8_W64", "S256_g2_W1024"])
def test_multi_token_decode_split(spec):
    """Every job split over two CTAs and merged through the workspace."""
    layer, prefix, new = spec
    c = ExtendCase([layer], prefix, new, seed=12, poison_tail=False, split="all")
    _store_chunk(c, 0)
    out, lse = _decode_multi(c, 0)
    assert_close(out, c.oracle(0), what="split multi-token decode")
    g = lse.double().cpu().numpy()
    assert np.all(np.abs(g - c.oracle_lse) <= 2e-3 * np.maximum(1.0, np.abs(c.oracle_lse)))
    assert c.fa.device_error() == 0


def test_one_new_token_equals_decode():
    """n_b = 1 for every sequence: the same attention as the single-token decode."""
    layer = lay(W.SLIDING, 256, 8, 1, 48)
    c = ExtendCase([layer], [40, 0, 100, 17], [1, 1, 1, 1], seed=13, poison_tail=False)
    _store_chunk(c, 0)
    out, _ = _decode_multi(c, 0)
    lens = torch.from_numpy((c.prefix + 1).astype(np.int32)).cuda()
    dout = torch.empty_like(out)
    n = c.cache.decode_workspace_bytes(0, c.B, int(lens.max()))
    ws = c.fa.workspace(n) if n else None
    c.cache.decode(0, c.q[0][: c.N], c.bt, lens, int(lens.max()), dout, None, ws)
    assert_close(out, dout.double().cpu().numpy(), what="multi-token vs decode")
    assert c.fa.device_error() == 0


def test_shared_layer_reads_the_source_slab():
    layers = [lay(W.SLIDING, 256, 8, 2, 64), lay(W.FULL, 512, 8, 1), lay(W.SLIDING, 256, 8, 2, 64, W.KV_AUTO)]
    c = ExtendCase(layers, [50, 130], [6, 3], seed=14, poison_tail=False)
    _store_chunk(c, 0)
    out, _ = _decode_multi(c, 2)
    assert_close(out, c.oracle(2), what="shared layer")
    assert c.fa.device_error() == 0
