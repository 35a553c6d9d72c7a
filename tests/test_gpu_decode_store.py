"""The fused store + decode call (fa_paged_decode_store_attn) against the two
separate calls it replaces and against the fp64 oracle.

The fused kernel writes the current token's rows with the same per-row code
as the store kernel and runs the same decode arithmetic, so outputs, lse and
slabs must equal the separate calls bit for bit; parity with the oracle then
follows from the decode tests, and is also checked directly on the
full-size E2B-like workload in the launch configuration the benchmark times.
"""
import numpy as np
import pytest
import torch

import workloads as W
from paged_case import DecodeCase, assert_close

pytestmark = pytest.mark.gpu


def lay(kind, D, hq, hkv, Wn=0, src=W.KV_OWN):
    return W.layer(kind, D, hq, hkv, Wn, src)


CASES = [
    # (layers, lens)
    ([lay(W.FULL, 512, 8, 1), lay(W.SLIDING, 256, 8, 1, 64), lay(W.SLIDING, 256, 8, 1, 64, W.KV_AUTO)],
     [1, 2, 15, 16, 17, 64, 65, 200, 513]),
    ([lay(W.SLIDING, 256, 16, 2, 33), lay(W.FULL, 256, 16, 2)], [3, 33, 34, 49, 150, 700]),
    ([lay(W.FULL, 512, 2, 2), lay(W.SLIDING, 512, 2, 2, 1)], [1, 5, 17, 40]),
]


def run_both(layers, lens, kv_dtype, seed, flags=0):
    sep = DecodeCase(layers, lens, 16, kv_dtype, seed=seed)
    fus = DecodeCase(layers, lens, 16, kv_dtype, seed=seed)
    if flags:
        sep.cache.set_flags(flags)
        fus.cache.set_flags(flags)
    sep.store_current()
    res_sep = [sep.decode(i) for i in range(len(layers))]
    res_fus = [fus.decode_store(i) for i in range(len(layers))]
    torch.cuda.synchronize()
    return sep, fus, res_sep, res_fus


@pytest.mark.parametrize("kv_dtype", [W.KV_BF16, W.KV_INT8, W.KV_FP8], ids=["bf16", "int8", "fp8"])
@pytest.mark.parametrize("ci", range(len(CASES)))
def test_fused_equals_store_then_decode(ci, kv_dtype):
    layers, lens = CASES[ci]
    sep, fus, rs, rf = run_both(layers, lens, kv_dtype, seed=21 + ci)
    for i, ((o1, l1), (o2, l2)) in enumerate(zip(rs, rf)):
        assert torch.equal(o1, o2), f"layer {i}: out differs"
        assert torch.equal(l1, l2), f"layer {i}: lse differs"
    for i in sep.slabs:
        for a, b in zip(sep.slabs[i], fus.slabs[i]):
            if a is not None:
                assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), f"slab of layer {i} differs"
    assert sep.fa.device_error() == 0


def test_fused_e2b_full_size_against_oracle_with_early_metadata():
    w = W.e2b_decode()
    case = DecodeCase(w.layers, W.seq_lens(w), w.page_size, w.kv_dtype, w.seed)
    case.cache.set_flags(case.fa.FLAG_EARLY_METADATA)
    seqs = [0, 1, 17, 40, 63]
    for i in range(len(case.layers)):
        out, lse = case.decode_store(i)
        ref, ref_lse = case.oracle_decode(i, seqs)
        assert_close(out[seqs], ref, what=f"fused layer {i}")
        g = lse[seqs].double().cpu().numpy()
        assert np.all(np.abs(g - ref_lse) <= 2e-3 * np.maximum(1.0, np.abs(ref_lse)))
    assert case.fa.device_error() == 0


def test_empty_sequence_row_is_still_stored_and_bad_slot_is_reported():
    layers = [lay(W.FULL, 256, 8, 1)]
    lens = [9, 0, 30]
    sep = DecodeCase(layers, lens, 16, W.KV_BF16, seed=5)
    fus = DecodeCase(layers, lens, 16, W.KV_BF16, seed=5)
    # sequence 1 has no context but a slot (on a page no sequence uses): both
    # paths store its row there
    bt = sep.plans[0].block_table
    free = sorted(set(range(sep.num_pages)) - set(bt[bt >= 0].tolist()))
    assert free
    page = free[0]
    slots = W.decode_slot_mapping(sep.lens, bt, 16)
    slots[1] = page * 16 + 3
    sl = torch.from_numpy(slots).cuda()
    k, v = sep.new_kv[0]
    sep.cache.store(0, k, v, sl)
    o1, l1 = sep.decode(0)
    o2, l2 = fus.decode_store(0, slots=sl)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(sep.slabs[0][0], fus.slabs[0][0]) and torch.equal(sep.slabs[0][1], fus.slabs[0][1])
    assert torch.equal(fus.slabs[0][0][page, 0, 3], k[1, 0])
    assert float(o2[1].abs().max()) == 0.0 and bool(torch.isinf(l2[1]).all())
    assert fus.fa.device_error() == 0
    # a slot past the pool is not stored and is reported
    bad = sl.clone()
    bad[2] = fus.num_pages * 16 + 5
    before = fus.slabs[0][0].clone()
    fus.decode_store(0, slots=bad)
    assert fus.fa.device_error() & fus.fa.DEV_ERR_SLOT
    assert torch.equal(before, fus.slabs[0][0])
