"""Multi-layer store and decode launches against the single-layer calls.

fa_kv_store_layers must leave every slab bit-identical to per-layer
fa_kv_store calls, and fa_paged_decode_attn_layers must give every layer the
same out and lse, bit for bit, as fa_paged_decode_attn on that layer (which
the other decode tests pin to the oracle); one case is also checked against
the oracle directly.
"""
import numpy as np
import pytest
import torch

import workloads as W
from paged_case import DecodeCase, assert_close

pytestmark = pytest.mark.gpu


def _groups(layers):
    return {d: [i for i, x in enumerate(layers) if x["head_dim"] == d] for d in (256, 512)}


def _decode_groups(case, lse=True):
    """Outputs of every layer from one multi-layer call per head_dim."""
    outs, lses = {}, {}
    for D, idx in _groups(case.layers).items():
        if not idx:
            continue
        o = [torch.full((case.B, case.layers[i]["num_q_heads"], D), float("nan"), dtype=torch.bfloat16,
                        device="cuda") for i in idx]
        l = [torch.full((case.B, case.layers[i]["num_q_heads"]), float("nan"), dtype=torch.float32, device="cuda")
             for i in idx] if lse else None
        n = case.cache.decode_layers_workspace_bytes(idx, case.B, case.max_len)
        ws = case.fa.workspace(n) if n else None
        case.cache.decode_layers(idx, [case.q[i] for i in idx], [case.bt_dev[i] for i in idx], case.lens_dev,
                                 case.max_len, o, l, ws)
        for k, i in enumerate(idx):
            outs[i] = o[k]
            lses[i] = l[k] if lse else None
    return outs, lses


@pytest.mark.parametrize("kv_dtype", [W.KV_BF16, W.KV_INT8, W.KV_FP8], ids=["bf16", "int8", "fp8"])
@pytest.mark.parametrize("lens", [[3, 33, 34, 49, 150, 700, 1, 517], [600] * 12 + [2049, 16, 17]],
                         ids=["mixed", "uniform"])
def test_layers_decode_equals_per_layer(kv_dtype, lens):
    layers = W.layout_12(8, 1, 64)
    case = DecodeCase(layers, lens, 16, kv_dtype, seed=5)
    case.store_current()
    ref = {i: case.decode(i) for i in range(len(layers))}
    outs, lses = _decode_groups(case)
    for i in range(len(layers)):
        assert torch.equal(outs[i], ref[i][0]), f"layer {i} out"
        assert torch.equal(lses[i], ref[i][1]), f"layer {i} lse"
    # a second call reuses the workspace (its counters were left zero)
    outs2, _ = _decode_groups(case, lse=False)
    for i in range(len(layers)):
        assert torch.equal(outs2[i], ref[i][0])
    assert case.fa.device_error() == 0


def test_layers_decode_matches_oracle_on_the_tiny_workload():
    """The tiny decode workload (a sliding, a full and a shared layer): the
    sliding layer and the layer sharing its slab go in one call."""
    w = W.tiny_decode()
    case = DecodeCase(w.layers, W.seq_lens(w), w.page_size, w.kv_dtype, w.seed, min_pool=w.min_pool_pages)
    assert case.src == [0, 1, 0]
    case.store_current()
    outs, lses = _decode_groups(case)
    for i in range(3):
        ref, ref_lse = case.oracle_decode(i, range(case.B))
        assert_close(outs[i], ref, what=f"layer {i}")
        assert np.all(np.abs(lses[i].double().cpu().numpy() - ref_lse) <= 2e-3 * np.maximum(1.0, np.abs(ref_lse)))
    assert case.fa.device_error() == 0


@pytest.mark.parametrize("kv_dtype", [W.KV_BF16, W.KV_INT8, W.KV_FP8], ids=["bf16", "int8", "fp8"])
def test_store_layers_equals_per_layer_stores(kv_dtype):
    import full_attention_gb300 as fa
    layers = W.layout_12(8, 1, 64)
    lens = [20, 33, 300, 17]
    a = DecodeCase(layers, lens, 16, kv_dtype, seed=7)
    b = DecodeCase(layers, lens, 16, kv_dtype, seed=7)
    a.store_current()
    owning = sorted(a.new_kv)
    all_layers = list(range(len(layers)))   # shared layers are skipped
    b.cache.store_layers(all_layers, [b.new_kv[i][0] if i in b.new_kv else None for i in all_layers],
                         [b.new_kv[i][1] if i in b.new_kv else None for i in all_layers],
                         [b.slot_mapping(i) for i in all_layers])
    torch.cuda.synchronize()
    for i in owning:
        for x, y in zip(a.slabs[i], b.slabs[i]):
            if x is not None:
                assert torch.equal(x.view(torch.uint8) if x.dtype != torch.uint8 else x,
                                   y.view(torch.uint8) if y.dtype != torch.uint8 else y), f"slab of layer {i}"
    assert fa.device_error() == 0


def test_layers_argument_errors():
    import full_attention_gb300 as fa
    layers = W.layout_12(8, 1, 64)
    case = DecodeCase(layers, [40, 70], 16, W.KV_BF16, seed=8)
    o = [torch.empty((2, 8, layers[i]["head_dim"]), dtype=torch.bfloat16, device="cuda") for i in (0, 4)]
    ws = case.fa.workspace(1 << 20)
    with pytest.raises(fa.FAError) as e:   # head_dims 256 and 512 in one call
        case.cache.decode_layers([0, 4], [case.q[0], case.q[4]], [case.bt_dev[0], case.bt_dev[4]], case.lens_dev,
                                 case.max_len, o, None, ws)
    assert e.value.status == fa.ERR_UNSUPPORTED
    with pytest.raises(fa.FAError) as e:   # a layer listed twice
        case.cache.decode_layers([0, 0], [case.q[0]] * 2, [case.bt_dev[0]] * 2, case.lens_dev, case.max_len,
                                 [o[0], o[0]], None, ws)
    assert e.value.status == fa.ERR_INVALID_ARG
    with pytest.raises(fa.FAError) as e:   # workspace too small
        case.cache.decode_layers([0, 1], [case.q[0], case.q[1]], [case.bt_dev[0], case.bt_dev[1]], case.lens_dev,
                                 case.max_len, [o[0], o[0].clone()], None, case.fa.workspace(16))
    assert e.value.status == fa.ERR_WORKSPACE
    # the reported size is enough (one wave of CTAs shared by the layers: at
    # most the per-layer workspaces end to end)
    n = case.cache.decode_layers_workspace_bytes([0, 1], 2, case.max_len)
    assert 0 < n <= sum((case.cache.decode_workspace_bytes(i, 2, case.max_len) + 255) // 256 * 256 for i in (0, 1))
    case.store_current()
    case.cache.decode_layers([0, 1], [case.q[0], case.q[1]], [case.bt_dev[0], case.bt_dev[1]], case.lens_dev,
                             case.max_len, [o[0], o[0].clone()], None, case.fa.workspace(n))
    assert fa.device_error() == 0
