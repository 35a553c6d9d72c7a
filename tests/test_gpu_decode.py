"""Decode parity: the CUDA path through the C ABI against the fp64 oracle.

Small cases compare every output; the full-size workloads compare sampled
sequences (every query head of each, every layer) in the launch
configuration the benchmark times.  Tolerance for bf16 outputs: max-abs
1e-2 and relative L2 2e-2 against the float64 oracle.
"""
import numpy as np
import pytest
import torch

import workloads as W
from paged_case import DecodeCase, assert_close

pytestmark = pytest.mark.gpu


def lay(kind, D, hq, hkv, Wn=0, src=W.KV_OWN):
    return W.layer(kind, D, hq, hkv, Wn, src)


def check_layers(case, seqs, layers=None, lse_tol=2e-3):
    case.store_current()
    for i in (range(len(case.layers)) if layers is None else layers):
        out, lse = case.decode(i)
        ref, ref_lse = case.oracle_decode(i, seqs)
        assert_close(out[list(seqs)], ref, what=f"layer {i}")
        g = lse[list(seqs)].double().cpu().numpy()
        assert np.all(np.abs(g - ref_lse) <= lse_tol * np.maximum(1.0, np.abs(ref_lse))), f"lse layer {i}"
    fa = case.fa
    assert fa.device_error() == 0


def test_tiny_decode_workload():
    w = W.tiny_decode()
    case = DecodeCase(w.layers, W.seq_lens(w), w.page_size, w.kv_dtype, w.seed, min_pool=w.min_pool_pages)
    assert case.src == [0, 1, 0]
    check_layers(case, range(case.B))


SMALL = [
    # (kind, D, hq, hkv, W, lens)
    (W.FULL, 512, 8, 1, 0, [1, 2, 15, 16, 17, 31, 33, 200, 513]),
    (W.SLIDING, 256, 8, 1, 64, [1, 16, 63, 64, 65, 66, 80, 81, 300]),
    (W.SLIDING, 256, 4, 1, 1, [1, 5, 17, 40]),
    (W.FULL, 256, 16, 2, 0, [7, 100, 257]),
    (W.SLIDING, 512, 2, 2, 33, [3, 33, 34, 49, 150]),
    (W.FULL, 512, 8, 8, 0, [20, 64]),
]


@pytest.mark.parametrize("kv_dtype", [W.KV_BF16, W.KV_INT8, W.KV_FP8], ids=["bf16", "int8", "fp8"])
@pytest.mark.parametrize("spec", SMALL, ids=[f"{'F' if s[0] == 0 else 'S'}{s[1]}_g{s[2] // s[3]}_W{s[4]}"
                                             for s in SMALL])
def test_small_decode(spec, kv_dtype):
    kind, D, hq, hkv, Wn, lens = spec
    layers = [lay(kind, D, hq, hkv, Wn), lay(kind, D, hq, hkv, Wn, W.KV_AUTO)]
    case = DecodeCase(layers, lens, 16, kv_dtype, seed=11, poison=(kv_dtype == W.KV_BF16))
    check_layers(case, range(case.B))


def test_page_size_32_and_zero_length():
    layers = [lay(W.SLIDING, 256, 8, 1, 40), lay(W.FULL, 512, 8, 1)]
    lens = [0, 1, 31, 32, 33, 95]
    case = DecodeCase(layers, [max(1, L) for L in lens], 32, seed=5)
    case.lens[0] = 0
    case.lens_dev[0] = 0
    case.store_current()
    for i in range(2):
        out, lse = case.decode(i)
        assert torch.all(out[0] == 0) and torch.all(torch.isinf(lse[0])) and torch.all(lse[0] < 0)
        ref, _ = case.oracle_decode(i, range(1, case.B))
        assert_close(out[1:], ref, what=f"layer {i}")


def test_window_one_is_exact_current_value():
    layers = [lay(W.SLIDING, 256, 8, 1, 1)]
    case = DecodeCase(layers, [1, 19, 64, 300], 16, seed=9)
    case.store_current()
    out, _ = case.decode(0)
    k, v = case.new_kv[0]
    assert torch.equal(out, v[:, :1, :].expand_as(out))


def test_constant_v_gives_constant_and_permutation_invariance():
    layers = [lay(W.FULL, 512, 8, 1)]
    case = DecodeCase(layers, [77, 160, 1000], 16, seed=4)
    case.store_current()
    out1, lse1 = case.decode(0)
    # permute physical pages: move every page p to perm[p], remap the table
    perm = torch.randperm(case.num_pages, generator=torch.Generator().manual_seed(3)).to("cuda")
    k_s, v_s, _, _ = case.slabs[0]
    k2 = torch.empty_like(k_s)
    v2 = torch.empty_like(v_s)
    k2[perm] = k_s
    v2[perm] = v_s
    k_s.copy_(k2)
    v_s.copy_(v2)
    bt = case.bt_dev[0]
    case.bt_dev[0] = torch.where(bt >= 0, perm[bt.clamp(min=0).long()].int(), bt)
    out2, lse2 = case.decode(0)
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)
    v_s.fill_(1.0)
    out3, _ = case.decode(0)
    assert torch.all(out3 == 1.0)


def test_determinism_and_graph_replay():
    w = W.e2b_decode()
    layers = w.layers[:5]
    case = DecodeCase(layers, W.seq_lens(w)[:16], 16, seed=1)
    case.store_current()
    outs = [case.decode(i) for i in range(5)]
    again = [case.decode(i) for i in range(5)]
    for (a, la), (b, lb) in zip(outs, again):
        assert torch.equal(a, b) and torch.equal(la, lb)


@pytest.mark.parametrize("kv_dtype", [W.KV_BF16, W.KV_INT8, W.KV_FP8], ids=["bf16", "int8", "fp8"])
@pytest.mark.parametrize("shape", ["d256_g8", "d256_g8_one_kv", "d512_g8"])
def test_repeated_decodes_are_bit_identical(shape, kv_dtype):
    """Alternating layers with many short segments per CTA (one-tile and
    three-tile units next to long ones) stress the per-segment hand-off of the
    queries: every repeat must equal the first run bit for bit."""
    if shape == "d256_g8":
        layers, lens = [lay(W.SLIDING, 256, 16, 2, 33), lay(W.FULL, 256, 16, 2)], [3, 33, 34, 49, 150, 700]
    elif shape == "d256_g8_one_kv":
        layers, lens = [lay(W.FULL, 256, 8, 1), lay(W.SLIDING, 256, 8, 1, 64)], [1, 17, 300, 1000, 5, 64, 65, 2049]
    else:
        layers, lens = [lay(W.SLIDING, 512, 8, 1, 40), lay(W.FULL, 512, 8, 1)], [3, 33, 34, 49, 150, 700]
    case = DecodeCase(layers, lens, 16, kv_dtype, seed=22)
    case.store_current()
    ref = [case.decode(i) for i in range(len(layers))]
    bad = 0
    for _ in range(60):
        for i in range(len(layers)):
            o, lse = case.decode(i)
            bad += not (torch.equal(o, ref[i][0]) and torch.equal(lse, ref[i][1]))
    assert bad == 0
    assert case.fa.device_error() == 0


def test_bad_page_id_sets_device_error():
    """A visible block-table entry outside the pool is skipped (the TMA box
    then lies outside the tensor and reads zeros) and reported."""
    layers = [lay(W.FULL, 512, 8, 1)]
    case = DecodeCase(layers, [40, 50], 16, seed=2)
    assert case.fa.device_error() == 0
    case.bt_dev[0][1, 1] = case.num_pages + 5
    case.decode(0)
    assert case.fa.device_error() & case.fa.DEV_ERR_PAGE
    case.bt_dev[0][1, 1] = -1
    case.decode(0)
    assert case.fa.device_error() & case.fa.DEV_ERR_PAGE
    assert case.fa.device_error() == 0


def test_length_past_max_seq_len_sets_device_error():
    """A sequence longer than the call's max_seq_len is cut to it and
    reported with FA_DEV_ERR_BOUND; within the bound nothing is reported."""
    layers = [lay(W.FULL, 512, 8, 1), lay(W.SLIDING, 256, 8, 1, 16)]
    case = DecodeCase(layers, [40, 50], 16, seed=2)
    assert case.fa.device_error() == 0
    real = case.max_len
    for i in range(len(layers)):
        case.max_len = 45            # the 50-token sequence is past it
        case.decode(i)
        assert case.fa.device_error() & case.fa.DEV_ERR_BOUND
        case.max_len = real
        case.decode(i)
        assert case.fa.device_error() == 0


# ------------------------------------------------------------------ full size
def _sample(B, n, seed):
    return sorted(np.random.default_rng(seed).choice(B, size=min(n, B), replace=False).tolist())


def test_e2b_decode_full_size():
    w = W.e2b_decode()
    case = DecodeCase(w.layers, W.seq_lens(w), w.page_size, w.kv_dtype, w.seed, poison=True)
    assert case.src[7:] == [6, 6, 4, 6, 6]
    lens = case.lens
    seqs = sorted(set(_sample(case.B, 5, 1) + [int(np.argmax(lens)), int(np.argmin(lens))]))
    check_layers(case, seqs)


def test_long_context_decode_full_size():
    """Contexts of 32k-131k tokens: the longest sequence is always checked (the
    split-K merges with the most partials), with both owning sliding layers,
    the owning full layer and shared layers of both kinds."""
    w = W.long_decode()
    case = DecodeCase(w.layers, W.seq_lens(w), w.page_size, w.kv_dtype, w.seed, window_table=True, poison=True)
    seqs = sorted(set(_sample(case.B, 3, 3) + [int(np.argmax(case.lens))]))
    check_layers(case, seqs, layers=[0, 4, 6, 7, 9, 11])


@pytest.mark.parametrize("make", [W.int8_decode, W.fp8_decode], ids=["int8", "fp8"])
def test_8bit_decode_full_size(make):
    w = make()
    case = DecodeCase(w.layers, W.seq_lens(w), w.page_size, w.kv_dtype, w.seed)
    lens = case.lens
    seqs = sorted(set(_sample(case.B, 4, 5) + [int(np.argmax(lens))]))
    check_layers(case, seqs)


def test_workspace_counters_left_zero_and_reusable():
    """Split units are merged by their last CTA through arrival counters at the
    head of the workspace; every call leaves them zero, so one buffer serves
    consecutive calls (and layers) with identical results."""
    w = W.e2b_decode()
    case = DecodeCase(w.layers[:5], W.seq_lens(w)[:32], 16, seed=6)
    case.store_current()
    n = max(case.cache.decode_workspace_bytes(i, case.B, case.max_len) for i in range(5))
    assert n > 0
    ws = case.fa.workspace(n)
    first = [case.decode(i, ws=ws) for i in range(5)]
    units = case.B * 1   # one KV head, 8 query heads: one unit per sequence
    assert int(ws[: units * 4].count_nonzero()) == 0
    again = [case.decode(i, ws=ws) for i in range(5)]
    for (a, la), (b, lb) in zip(first, again):
        assert torch.equal(a, b) and torch.equal(la, lb)
    assert case.fa.device_error() == 0


def test_early_metadata_flag_gives_identical_results():
    """Reading the index arrays before the preceding kernel finishes changes
    only when they are read, never what is computed."""
    w = W.e2b_decode()
    case = DecodeCase(w.layers, W.seq_lens(w)[:24], 16, seed=8)
    case.store_current()
    plain = [case.decode(i) for i in range(len(case.layers))]
    case.cache.set_flags(case.fa.FLAG_EARLY_METADATA)
    case.store_current()
    early = [case.decode(i) for i in range(len(case.layers))]
    for (a, la), (b, lb) in zip(plain, early):
        assert torch.equal(a, b) and torch.equal(la, lb)
    assert case.fa.device_error() == 0


@pytest.mark.parametrize("kv_dtype", [W.KV_BF16, W.KV_INT8, W.KV_FP8], ids=["bf16", "int8", "fp8"])
def test_window_pool(kv_dtype):
    """Sliding layers on a pool of their own: their tables hold only the
    in-window pages (-1 elsewhere) and index a pool sized for the windows,
    while the full layer keeps the big pool; a shared sliding layer reads
    its source's window-pool slab."""
    layers = [lay(W.SLIDING, 256, 8, 1, 64), lay(W.FULL, 512, 8, 1), lay(W.SLIDING, 256, 8, 1, 64, W.KV_AUTO)]
    lens = [3000, 17, 1024, 4500, 65, 2]
    case = DecodeCase(layers, lens, 16, kv_dtype, seed=15, window_table=True, window_pool=True,
                      poison=(kv_dtype == W.KV_BF16))
    assert case.window_pages < case.num_pages // 10
    assert case.slabs[0][0].shape[0] == case.window_pages and case.slabs[1][0].shape[0] == case.num_pages
    check_layers(case, range(case.B))
    # the extend kernel on the same pool: one new token per sequence, keys from the slab
    q = case.q[0]
    out = torch.empty_like(q)
    indptr = torch.arange(0, case.B + 1, dtype=torch.int32, device="cuda")
    case.cache.decode_multi(0, q, indptr, case.lens_dev, case.bt_dev[0], 1, case.max_len, out)
    ref, _ = case.oracle_decode(0, range(case.B))
    assert_close(out, ref, what="multi-token decode on the window pool")
    # a page id past the window pool (not past the full pool) is refused by the sliding layer
    bt = case.bt_dev[0].clone()
    L0 = int(case.lens[0])
    bt[0, (L0 - 1) // 16] = case.window_pages
    out = torch.empty_like(q)
    ws = case.workspace(0)
    case.cache.decode(0, q, bt, case.lens_dev, case.max_len, out, None, ws)
    assert case.fa.device_error() & case.fa.DEV_ERR_PAGE
