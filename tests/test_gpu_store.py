"""Paged KV store parity: fa_kv_store against the oracle's store, bit for bit.

Every format (bf16 copy, int8 and fp8 e4m3 per-token-head codes with fp32
scales), both head dims, one and two KV heads.  The rows mix seeded normals
with rows built to hit the rounding rules: an all-zero row, a row of -0.0,
rows whose largest magnitude is 448 or 127 (scale exactly 1, so the codes
are the values rounded, ties included), and rows spanning 2^-20 .. 2^4 (e4m3
subnormals and flushes to zero).  Slots include padding (-1); slots the
store does not write keep their prior contents.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu

FORMATS = [W.KV_BF16, W.KV_INT8, W.KV_FP8]
FORMAT_IDS = ["bf16", "int8", "fp8"]


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _rows(T, H, D, seed):
    """bf16 rows [T][H][D]: normals plus rows aimed at the rounding rules."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((T, H, D), generator=g) * 2.0
    x[1, 0] = 0.0
    x[2, H - 1] = -0.0
    ties = torch.tensor([448, 1.0625, 1.1875, 432, -3, 2 ** -10, 3 * 2 ** -10, 15 * 2 ** -10, -(2 ** -10), 2.5,
                         3.5, -2.5, 0.5, 126.5, 127, -127])
    x[3, 0] = ties.repeat(D // ties.numel() + 1)[:D]
    e = torch.randint(-20, 5, (D,), generator=g).float()
    x[4, H - 1] = torch.sign(torch.randn(D, generator=g)) * torch.exp2(e)
    x[5, 0, :] = 127.0 * torch.sign(torch.randn(D, generator=g)) * torch.rand(D, generator=g)
    x[5, 0, 7] = 127.0
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("kv_dtype", FORMATS, ids=FORMAT_IDS)
@pytest.mark.parametrize("D,H", [(256, 1), (512, 1), (256, 2), (512, 2)])
def test_store_matches_oracle_bit_for_bit(kv_dtype, D, H):
    import full_attention_gb300 as fa
    ps, pool, T = 16, 9, 40
    cache = fa.Cache([W.layer(W.FULL, D, 8, H)], pool, ps, kv_dtype)
    k_s, v_s, ks_s, vs_s = cache.allocate("cuda")[0]
    # prior contents of every slot (unwritten slots must keep them)
    gen = torch.Generator(device="cuda").manual_seed(3)
    if kv_dtype == W.KV_BF16:
        k_s.copy_(torch.randn(k_s.shape, generator=gen, device="cuda").to(torch.bfloat16))
        v_s.copy_(torch.randn(v_s.shape, generator=gen, device="cuda").to(torch.bfloat16))
    else:
        k_s.copy_(torch.randint(-100, 100, k_s.shape, generator=gen, device="cuda").to(k_s.dtype))
        v_s.copy_(torch.randint(-100, 100, v_s.shape, generator=gen, device="cuda").to(v_s.dtype))
        ks_s.fill_(0.25)
        vs_s.fill_(0.5)
    k = _rows(T, H, D, 10).cuda()
    v = _rows(T, H, D, 11).cuda()
    slots = np.random.default_rng(4).permutation(pool * ps)[:T].astype(np.int32)
    slots[[6, 17, 30]] = -1
    before = [t.clone() for t in (k_s, v_s, ks_s, vs_s) if t is not None]
    cache.store(0, k, v, torch.from_numpy(slots).cuda())
    torch.cuda.synchronize()
    assert fa.device_error() == 0

    if kv_dtype == W.KV_BF16:
        ok, ov = _bits(before[0]), _bits(before[1])
        oracle.store_bf16(ok, ov, _bits(k), _bits(v), slots, ps)
        assert np.array_equal(_bits(k_s), ok) and np.array_equal(_bits(v_s), ov)
        return
    ck, cv = before[0].cpu().numpy(), before[1].cpu().numpy()
    sk, sv = before[2].cpu().numpy(), before[3].cpu().numpy()
    store = oracle.store_fp8 if kv_dtype == W.KV_FP8 else oracle.store_int8
    store(ck, cv, sk, sv, _bits(k), _bits(v), slots, ps)
    assert np.array_equal(k_s.cpu().numpy(), ck) and np.array_equal(v_s.cpu().numpy(), cv)
    assert np.array_equal(ks_s.cpu().numpy().view(np.uint32), sk.view(np.uint32))
    assert np.array_equal(vs_s.cpu().numpy().view(np.uint32), sv.view(np.uint32))
    if kv_dtype == W.KV_FP8:
        codes = k_s.cpu().numpy()
        for slot in slots[slots >= 0]:
            row = codes[slot // ps, :, slot % ps]
            assert not np.any((row & 0x7F) == 0x7F), "the store never writes a NaN code"
