"""The allocation-free decode entry point against the regular one.

Some callers cannot allocate device memory: a plugin inside a serving
framework that hands out no allocator, or an engine that reserves its memory
budget at start-up and forbids cudaMalloc on the hot path.  For them
fa_paged_decode_attn_noalloc runs the same decode with the library's fixed
scratch array instead of a caller workspace.  These tests call it through the
C ABI twice in a row and compare each result with fa_paged_decode_attn's, and
check that a call needing more scratch than the fixed array is refused.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test.
"""
import pytest
import torch

import workloads as W
from paged_case import DecodeCase, assert_close

pytestmark = pytest.mark.gpu


def test_noalloc_decode_matches_regular_decode_twice():
    w = W.e2b_decode()
    case = DecodeCase(w.layers[:5], W.seq_lens(w)[:48], 16, seed=12)
    case.store_current()
    fa = case.fa
    for i in range(len(case.layers)):
        # the split-K scratch is really used: the plan splits these sequences
        assert case.cache.decode_workspace_bytes(i, case.B, case.max_len) > 0
        ref_out, ref_lse = case.decode(i)
        d = case.layers[i]
        for _ in range(2):   # the second call reuses the scratch the first one left
            out = torch.full((case.B, d["num_q_heads"], d["head_dim"]), float("nan"), dtype=torch.bfloat16,
                             device="cuda")
            lse = torch.full((case.B, d["num_q_heads"]), float("nan"), dtype=torch.float32, device="cuda")
            case.cache.decode_noalloc(i, case.q[i], case.bt_dev[i], case.lens_dev, case.max_len, out, lse)
            torch.cuda.synchronize()
            # the same kernel and plan as the regular call: bit for bit the same
            # result (within the float tolerance a fortiori), whatever stale
            # contents the scratch held
            assert_close(out, ref_out.double().cpu().numpy(), what=f"no-alloc layer {i}")
            assert torch.equal(out, ref_out), f"no-alloc layer {i}: output differs from the regular call"
            assert torch.equal(lse, ref_lse), f"no-alloc layer {i}: lse differs from the regular call"
    assert fa.device_error() == 0


def test_noalloc_decode_refuses_scratch_beyond_its_maximum():
    fa = pytest.importorskip("full_attention_gb300")
    layers = [W.layer(W.FULL, 512, 8, 1)]
    cache = fa.Cache(layers, 64, 16)
    cache.allocate()
    B, max_len = 4096, 4096
    need = cache.decode_workspace_bytes(0, B, max_len)
    assert need > fa.NOALLOC_SCRATCH_BYTES
    q = torch.zeros((B, 8, 512), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((B, max_len // 16), dtype=torch.int32, device="cuda")
    lens = torch.ones(B, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    with pytest.raises(fa.FAError) as e:
        cache.decode_noalloc(0, q, bt, lens, max_len, out)
    assert e.value.status == fa.ERR_WORKSPACE
    assert fa.device_error() == 0
