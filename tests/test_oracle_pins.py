"""Pins of the fp64 oracle against things other than itself.

* dense attention computed by a library routine (torch SDPA in float64 with an
  explicit boolean mask) and by a hand-written triple loop, on tiny unpaged
  inputs that the test pages itself;
* closed forms (W = 1, q = 0, constant V, one key, two keys);
* invariants (physical page permutation, W >= L, shared == copied slab,
  softmax rows sum to 1, chunked == one-shot extend, decode == extend row,
  sliding != full once L > W);
* the per-token byte counts, slab counts, sources and ratios the pages print;
* int8 codes against exact rational rounding and hand-worked ties;
* fp8 e4m3 codes against hand-worked values and ties, torch's float8_e4m3fn
  cast (a library routine), and a value table built here from the format's
  definition with exact rationals.

A planted-mistake test at the end checks that plausible slips in the oracle
(window off by one, scale dropped, page offset misread, K and V swapped) make
at least one of these pins fail.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import FULL, SLIDING, KV_AUTO, KV_OWN

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# helpers written independently of the oracle
# ---------------------------------------------------------------------------

def f32_to_bf16_bits(x):
    """Round float32 values to bf16 bit patterns (test-side input helper)."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16) \
        .to(torch.float64).numpy()


def lay(kind, D, hq, hkv, W=0, src=KV_OWN):
    return dict(kind=kind, head_dim=D, num_q_heads=hq, num_kv_heads=hkv,
                window=W if kind == SLIDING else 0, kv_source=src,
                sm_scale=float(np.float32(1.0 / math.sqrt(D))))


def page_dense(dense_k, dense_v, page_size, rng, extra_pages=3):
    """dense [L][Hkv][D] bf16 bits -> (slab_k, slab_v, block_table_row) with a
    random physical page order.  Written here, not taken from the oracle."""
    L, H, D = dense_k.shape
    npg = (L + page_size - 1) // page_size
    pool = npg + extra_pages
    perm = rng.permutation(pool)
    sk = np.zeros((pool, H, page_size, D), dtype=np.uint16)
    sv = np.zeros_like(sk)
    for pos in range(L):
        sk[perm[pos // page_size], :, pos % page_size, :] = dense_k[pos]
        sv[perm[pos // page_size], :, pos % page_size, :] = dense_v[pos]
    return sk, sv, perm[:npg].astype(np.int32)


def sdpa_dense(q, k, v, q_pos, kind, W, scale):
    """Library attention: q [n][D], k,v [L][D] float64, explicit bool mask."""
    L = k.shape[0]
    kp = np.arange(L)[None, :]
    qp = np.asarray(q_pos)[:, None]
    mask = kp <= qp
    if kind == SLIDING:
        mask &= (qp - kp) < W
    out = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(k)[None], torch.from_numpy(v)[None],
        attn_mask=torch.from_numpy(mask)[None], scale=scale)
    return out[0].numpy()


def loop_attention(q, k, v, q_pos, kind, W, scale):
    """Triple-loop textbook masked softmax (brute force, tiny inputs only)."""
    out = np.zeros((len(q_pos), k.shape[1]))
    for i, qp in enumerate(q_pos):
        keys = [t for t in range(k.shape[0])
                if t <= qp and (kind == FULL or qp - t < W)]
        s = [scale * sum(q[i, d] * k[t, d] for d in range(k.shape[1])) for t in keys]
        mx = max(s)
        w = [math.exp(x - mx) for x in s]
        z = sum(w)
        for d in range(k.shape[1]):
            out[i, d] = sum(wi * v[t, d] for wi, t in zip(w, keys)) / z
    return out


def rand_bits(rng, shape, scale=1.0):
    return f32_to_bf16_bits(rng.standard_normal(shape).astype(np.float32) * scale)


# ---------------------------------------------------------------------------
# pins, as functions of an oracle module (so a mutated oracle can be checked)
# ---------------------------------------------------------------------------

def pin_decode_vs_dense(orc, seed=0):
    rng = np.random.default_rng(seed)
    for ps, L, kind, W, D, hq, hkv in [(1, 7, SLIDING, 3, 8, 2, 1), (4, 19, FULL, 0, 16, 4, 2),
                                       (16, 40, SLIDING, 9, 16, 4, 1), (4, 13, SLIDING, 64, 8, 2, 2),
                                       (16, 33, FULL, 0, 32, 8, 1)]:
        dk, dv = rand_bits(rng, (L, hkv, D)), rand_bits(rng, (L, hkv, D))
        sk, sv, bt = page_dense(dk, dv, ps, rng)
        q = rand_bits(rng, (1, hq, D))
        layers = [lay(kind, D, hq, hkv, W)]
        out, lse = orc.paged_decode(layers, 0, {0: (sk, sv)}, q, bt[None], np.array([L]), ps)
        g = hq // hkv
        for j in range(hq):
            h = j // g
            ref = sdpa_dense(bits_to_f64(q[0, j])[None], bits_to_f64(dk[:, h]), bits_to_f64(dv[:, h]),
                             [L - 1], kind, W, layers[0]["sm_scale"])[0]
            np.testing.assert_allclose(out[0, j], ref, rtol=0, atol=1e-12)


def pin_decode_vs_loops(orc, seed=1):
    rng = np.random.default_rng(seed)
    for ps, L, kind, W in [(4, 11, SLIDING, 5), (2, 6, FULL, 0), (4, 9, SLIDING, 1)]:
        D = 4
        dk, dv = rand_bits(rng, (L, 1, D)), rand_bits(rng, (L, 1, D))
        sk, sv, bt = page_dense(dk, dv, ps, rng)
        q = rand_bits(rng, (1, 1, D))
        layers = [lay(kind, D, 1, 1, W)]
        out, _ = orc.paged_decode(layers, 0, {0: (sk, sv)}, q, bt[None], np.array([L]), ps)
        ref = loop_attention(bits_to_f64(q[0]), bits_to_f64(dk[:, 0]), bits_to_f64(dv[:, 0]),
                             [L - 1], kind, W, layers[0]["sm_scale"])
        np.testing.assert_allclose(out[0], ref, rtol=0, atol=1e-12)


def pin_extend_vs_dense(orc, seed=2):
    rng = np.random.default_rng(seed)
    for ps, kind, W, D, hq, hkv, pref, chunk in [(4, SLIDING, 6, 8, 4, 2, [9, 0, 4], [5, 3, 0]),
                                                 (16, FULL, 0, 16, 2, 1, [17, 32], [12, 1]),
                                                 (1, SLIDING, 3, 8, 2, 1, [5], [6])]:
        layers = [lay(kind, D, hq, hkv, W)]
        B = len(pref)
        total = [p + c for p, c in zip(pref, chunk)]
        dense_k = [rand_bits(rng, (t, hkv, D)) for t in total]
        dense_v = [rand_bits(rng, (t, hkv, D)) for t in total]
        maxp = max((p + ps - 1) // ps for p in pref) + 1
        pool = sum((p + ps - 1) // ps for p in pref) + 2
        perm = rng.permutation(pool)
        sk = np.zeros((pool, hkv, ps, D), np.uint16)
        sv = np.zeros_like(sk)
        bt = np.full((B, maxp), -1, np.int32)
        k = 0
        for b in range(B):
            for lp in range((pref[b] + ps - 1) // ps):
                bt[b, lp] = perm[k]
                k += 1
            for pos in range(pref[b]):
                sk[bt[b, pos // ps], :, pos % ps] = dense_k[b][pos]
                sv[bt[b, pos // ps], :, pos % ps] = dense_v[b][pos]
        indptr = np.concatenate([[0], np.cumsum(chunk)]).astype(np.int32)
        q = rand_bits(rng, (indptr[-1], hq, D))
        kx = np.concatenate([dense_k[b][pref[b]:] for b in range(B)]) if indptr[-1] else \
            np.zeros((0, hkv, D), np.uint16)
        vx = np.concatenate([dense_v[b][pref[b]:] for b in range(B)]) if indptr[-1] else \
            np.zeros((0, hkv, D), np.uint16)
        out, _ = orc.paged_extend(layers, 0, {0: (sk, sv)}, q, kx, vx, indptr, np.array(pref), bt, ps)
        g = hq // hkv
        for b in range(B):
            if chunk[b] == 0:
                continue
            for j in range(hq):
                h = j // g
                qq = bits_to_f64(q[indptr[b]:indptr[b + 1], j])
                ref = sdpa_dense(qq, bits_to_f64(dense_k[b][:, h]), bits_to_f64(dense_v[b][:, h]),
                                 np.arange(pref[b], total[b]), kind, W, layers[0]["sm_scale"])
                np.testing.assert_allclose(out[indptr[b]:indptr[b + 1], j], ref, rtol=0, atol=1e-12)


def pin_window_one_is_current_value(orc, seed=3):
    rng = np.random.default_rng(seed)
    ps, L, D = 4, 10, 8
    dk, dv = rand_bits(rng, (L, 1, D)), rand_bits(rng, (L, 1, D))
    sk, sv, bt = page_dense(dk, dv, ps, rng)
    q = rand_bits(rng, (1, 2, D))
    out, _ = orc.paged_decode([lay(SLIDING, D, 2, 1, 1)], 0, {0: (sk, sv)}, q, bt[None],
                              np.array([L]), ps)
    for j in range(2):
        assert np.array_equal(out[0, j], bits_to_f64(dv[L - 1, 0]))


def pin_zero_query_is_mean(orc, seed=4):
    rng = np.random.default_rng(seed)
    ps, L, D, W = 4, 23, 8, 7
    dk, dv = rand_bits(rng, (L, 1, D)), rand_bits(rng, (L, 1, D))
    sk, sv, bt = page_dense(dk, dv, ps, rng)
    q = np.zeros((1, 1, D), np.uint16)
    for kind, lo in [(SLIDING, L - W), (FULL, 0)]:
        out, lse = orc.paged_decode([lay(kind, D, 1, 1, W)], 0, {0: (sk, sv)}, q, bt[None],
                                    np.array([L]), ps)
        ref = bits_to_f64(dv[lo:L, 0]).mean(axis=0)
        np.testing.assert_allclose(out[0, 0], ref, rtol=0, atol=1e-14)
        assert abs(lse[0, 0] - math.log(L - lo)) < 1e-12


def pin_constant_v_and_single_key(orc, seed=5):
    rng = np.random.default_rng(seed)
    ps, D = 4, 8
    L = 13
    dk = rand_bits(rng, (L, 1, D))
    c = rand_bits(rng, (1, 1, D))
    dv = np.repeat(c, L, axis=0)
    sk, sv, bt = page_dense(dk, dv, ps, rng)
    q = rand_bits(rng, (1, 1, D))
    out, _ = orc.paged_decode([lay(FULL, D, 1, 1)], 0, {0: (sk, sv)}, q, bt[None], np.array([L]), ps)
    np.testing.assert_allclose(out[0, 0], bits_to_f64(c[0, 0]), rtol=0, atol=1e-14)
    # a single key: the output is that key's value row
    out, lse = orc.paged_decode([lay(FULL, D, 1, 1)], 0, {0: (sk, sv)}, q, bt[None], np.array([1]), ps)
    assert np.array_equal(out[0, 0], bits_to_f64(dv[0, 0]))
    s0 = lay(FULL, D, 1, 1)["sm_scale"] * float(bits_to_f64(q[0, 0]) @ bits_to_f64(dk[0, 0]))
    assert abs(lse[0, 0] - s0) < 1e-12


def pin_two_keys(orc, seed=6):
    rng = np.random.default_rng(seed)
    ps, D = 1, 4
    dk, dv = rand_bits(rng, (2, 1, D)), rand_bits(rng, (2, 1, D))
    sk, sv, bt = page_dense(dk, dv, ps, rng)
    q = rand_bits(rng, (1, 1, D))
    ly = lay(FULL, D, 1, 1)
    out, _ = orc.paged_decode([ly], 0, {0: (sk, sv)}, q, bt[None], np.array([2]), ps)
    qv = bits_to_f64(q[0, 0])
    s0 = ly["sm_scale"] * float(qv @ bits_to_f64(dk[0, 0]))
    s1 = ly["sm_scale"] * float(qv @ bits_to_f64(dk[1, 0]))
    w1 = 1.0 / (1.0 + math.exp(s0 - s1))     # sigmoid(s1 - s0)
    ref = (1 - w1) * bits_to_f64(dv[0, 0]) + w1 * bits_to_f64(dv[1, 0])
    np.testing.assert_allclose(out[0, 0], ref, rtol=0, atol=1e-14)


def pin_sliding_differs_from_full(orc, seed=7):
    rng = np.random.default_rng(seed)
    ps, L, D, W = 4, 30, 8, 8
    dk, dv = rand_bits(rng, (L, 1, D)), rand_bits(rng, (L, 1, D))
    sk, sv, bt = page_dense(dk, dv, ps, rng)
    q = rand_bits(rng, (1, 1, D))
    a, _ = orc.paged_decode([lay(SLIDING, D, 1, 1, W)], 0, {0: (sk, sv)}, q, bt[None], np.array([L]), ps)
    b, _ = orc.paged_decode([lay(FULL, D, 1, 1)], 0, {0: (sk, sv)}, q, bt[None], np.array([L]), ps)
    assert np.max(np.abs(a - b)) > 1e-3
    c, _ = orc.paged_decode([lay(SLIDING, D, 1, 1, L)], 0, {0: (sk, sv)}, q, bt[None], np.array([L]), ps)
    assert np.array_equal(c, b)


def pin_page_permutation(orc, seed=8):
    rng = np.random.default_rng(seed)
    ps, L, D = 4, 21, 8
    dk, dv = rand_bits(rng, (L, 2, D)), rand_bits(rng, (L, 2, D))
    sk, sv, bt = page_dense(dk, dv, ps, rng)
    q = rand_bits(rng, (1, 4, D))
    ly = [lay(SLIDING, D, 4, 2, 11)]
    a, la = orc.paged_decode(ly, 0, {0: (sk, sv)}, q, bt[None], np.array([L]), ps)
    perm = rng.permutation(sk.shape[0])
    inv = np.argsort(perm)
    sk2, sv2 = sk[inv], sv[inv]          # page p moves to slot perm[p]
    bt2 = perm[bt].astype(np.int32)
    b, lb = orc.paged_decode(ly, 0, {0: (sk2, sv2)}, q, bt2[None], np.array([L]), ps)
    assert np.array_equal(a, b) and np.array_equal(la, lb)


def pin_shared_equals_copy(orc, seed=9):
    rng = np.random.default_rng(seed)
    ps, L, D = 4, 17, 8
    dk, dv = rand_bits(rng, (L, 1, D)), rand_bits(rng, (L, 1, D))
    sk, sv, bt = page_dense(dk, dv, ps, rng)
    q = rand_bits(rng, (1, 2, D))
    layers = [lay(SLIDING, D, 2, 1, 6), lay(FULL, D, 2, 1), lay(SLIDING, D, 2, 1, 6, KV_AUTO)]
    junk = rand_bits(rng, sk.shape)
    slabs = {0: (sk, sv), 1: (junk, junk)}
    a, _ = orc.paged_decode(layers, 2, slabs, q, bt[None], np.array([L]), ps)
    solo = [lay(SLIDING, D, 2, 1, 6)]
    b, _ = orc.paged_decode(solo, 0, {0: (sk.copy(), sv.copy())}, q, bt[None], np.array([L]), ps)
    assert np.array_equal(a, b)


def pin_probabilities_sum_to_one(orc, seed=10):
    rng = np.random.default_rng(seed)
    for n in [1, 2, 17, 300]:
        K = rng.standard_normal((n, 16)) * 3
        V = rng.standard_normal((n, 16))
        q = rng.standard_normal(16)
        _, _, p = orc.softmax_attention(q, K, V, 0.25)
        assert abs(p.sum() - 1.0) < 1e-12 and np.all(p >= 0)


def pin_chunked_equals_one_shot(orc, seed=11):
    """Extend over one prompt in chunks == one shot == decode at each position."""
    rng = np.random.default_rng(seed)
    ps, D, T = 4, 8, 26
    for kind, W in [(SLIDING, 7), (FULL, 0)]:
        ly = [lay(kind, D, 2, 1, W)]
        dk, dv = rand_bits(rng, (T, 1, D)), rand_bits(rng, (T, 1, D))
        q = rand_bits(rng, (T, 2, D))
        pool = (T + ps - 1) // ps + 2
        perm = rng.permutation(pool).astype(np.int32)
        bt = perm[None, : (T + ps - 1) // ps].copy()
        sk = np.zeros((pool, 1, ps, D), np.uint16)
        sv = np.zeros_like(sk)
        one, _ = orc.paged_extend(ly, 0, {0: (sk, sv)}, q, dk, dv, np.array([0, T]), np.array([0]), bt, ps)
        chunks = []
        for c0 in range(0, T, 6):
            c1 = min(T, c0 + 6)
            part, _ = orc.paged_extend(ly, 0, {0: (sk, sv)}, q[c0:c1], dk[c0:c1], dv[c0:c1],
                                       np.array([0, c1 - c0]), np.array([c0]), bt, ps)
            chunks.append(part)
            orc.store_bf16(sk, sv, dk[c0:c1], dv[c0:c1],
                           [int(bt[0, p // ps]) * ps + p % ps for p in range(c0, c1)], ps)
        np.testing.assert_allclose(np.concatenate(chunks), one, rtol=0, atol=1e-13)
        for pos in [0, 5, T - 1]:
            dec, _ = orc.paged_decode(ly, 0, {0: (sk, sv)}, q[pos][None], bt, np.array([pos + 1]), ps)
            np.testing.assert_allclose(dec[0], one[pos], rtol=0, atol=1e-13)


PINS = [pin_decode_vs_dense, pin_decode_vs_loops, pin_extend_vs_dense, pin_window_one_is_current_value,
        pin_zero_query_is_mean, pin_constant_v_and_single_key, pin_two_keys,
        pin_sliding_differs_from_full, pin_page_permutation, pin_shared_equals_copy,
        pin_probabilities_sum_to_one, pin_chunked_equals_one_shot]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_attention_pin(pin):
    pin(oracle)


# ---------------------------------------------------------------------------
# store pins
# ---------------------------------------------------------------------------

def test_store_bf16_gather_roundtrip():
    rng = np.random.default_rng(20)
    ps, T, H, D, pool = 16, 50, 2, 32, 9
    k, v = rand_bits(rng, (T, H, D)), rand_bits(rng, (T, H, D))
    slots = rng.permutation(pool * ps)[:T].astype(np.int32)
    slots[7] = -1
    sk = np.zeros((pool, H, ps, D), np.uint16)
    sv = np.zeros_like(sk)
    oracle.store_bf16(sk, sv, k, v, slots, ps)
    for t in range(T):
        if slots[t] < 0:
            continue
        bt_row = np.arange(pool, dtype=np.int32)     # identity table: position == slot
        for h in range(H):
            got = oracle.gather_rows(sk, None, bt_row, [slots[t]], h, ps)[0]
            assert np.array_equal(got, bits_to_f64(k[t, h]))
            got = oracle.gather_rows(sv, None, bt_row, [slots[t]], h, ps)[0]
            assert np.array_equal(got, bits_to_f64(v[t, h]))
    # the skipped token wrote nothing: exactly T-1 rows per head are non-zero
    assert int(np.count_nonzero(np.any(sk != 0, axis=-1))) == (T - 1) * H


def read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def test_int8_ties_golden():
    g = {r[0]: r[1:] for r in read_golden("int8_ties.txt")}
    x = np.array([float(t) for t in g["x"]], np.float32)
    bits = f32_to_bf16_bits(x)
    assert np.array_equal(bits_to_f64(bits), x.astype(np.float64))   # all exact in bf16
    c, s = oracle.quantize_int8_per_token_head(bits[None])
    assert float(s[0]) == float(g["scale"][0])
    assert c[0].tolist() == [int(t) for t in g["codes"]]


def test_int8_codes_match_exact_rational_rounding():
    """Away from ties, fp32 x / fl(a/127) rounds like the exact 127 x / a."""
    rng = np.random.default_rng(21)
    x = f32_to_bf16_bits(rng.standard_normal((64, 256)).astype(np.float32) * 2.0)
    c, s = oracle.quantize_int8_per_token_head(x)
    xs = bits_to_f64(x)
    checked = 0
    for r in range(x.shape[0]):
        a = max(Fraction(float(t)).__abs__() for t in xs[r])
        for d in range(x.shape[1]):
            exact = Fraction(127) * Fraction(float(xs[r, d])) / a
            frac = exact - math.floor(exact)
            if abs(frac - Fraction(1, 2)) < Fraction(1, 10000):
                continue
            assert int(c[r, d]) == round(exact)
            checked += 1
        # the absmax element maps to +-127 and the reconstruction error is <= s/2
        assert np.max(np.abs(c[r].astype(int))) == 127
        err = np.abs(xs[r] - c[r].astype(np.float64) * float(s[r]))
        # x / s is rounded to fp32 before rint: half an ulp at 127 is 2**-18
        assert np.all(err <= float(s[r]) * (0.5 + 2.0 ** -18) * (1 + 1e-12))
        assert float(s[r]) == float(np.float32(np.float32(a) / np.float32(127)))
    assert checked > 0.99 * x.size


def test_int8_zero_row_and_store():
    rng = np.random.default_rng(22)
    ps, T, H, D, pool = 4, 6, 2, 16, 5
    k, v = rand_bits(rng, (T, H, D)), rand_bits(rng, (T, H, D))
    k[2, 1] = 0
    v[4, 0] = 0x8000          # -0.0 everywhere: absmax 0
    c, s = oracle.quantize_int8_per_token_head(k)
    assert s[2, 1] == 0 and np.all(c[2, 1] == 0)
    slots = np.array([0, 5, 6, -1, 19, 11], np.int32)
    ck = np.zeros((pool, H, ps, D), np.int8)
    cv = np.zeros_like(ck)
    sk = np.zeros((pool, H, ps), np.float32)
    sv = np.zeros_like(sk)
    oracle.store_int8(ck, cv, sk, sv, k, v, slots, ps)
    assert sv[4, 0, 3] == 0 and np.all(cv[4, 0, 3] == 0)
    for t, slot in enumerate(slots):
        if slot < 0:
            continue
        p, o = divmod(int(slot), ps)
        c1, s1 = oracle.quantize_int8_per_token_head(k[t])
        assert np.array_equal(ck[p, :, o], c1) and np.array_equal(sk[p, :, o], s1)
    # dequantised gather lands within s/2 of every input value
    bt_row = np.arange(pool, dtype=np.int32)
    for t, slot in enumerate(slots):
        if slot < 0:
            continue
        for h in range(H):
            got = oracle.gather_rows(ck, sk, bt_row, [slot], h, ps)[0]
            assert np.all(np.abs(got - bits_to_f64(k[t, h])) <= sk[slot // ps, h, slot % ps] / 2 + 1e-12)


# ---------------------------------------------------------------------------
# fp8 e4m3 pins
# ---------------------------------------------------------------------------

def e4m3_table_exact():
    """Every finite non-negative e4m3 value as an exact rational, by code,
    built from the format's definition (bias 7, 3 mantissa bits, exponent 0
    subnormal, code 0x7F NaN)."""
    out = {}
    for code in range(0x7F):
        e, m = code >> 3, code & 7
        out[code] = Fraction(m, 8) * Fraction(1, 64) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
    return out


def e4m3_nearest_exact(y: Fraction) -> int:
    """Code of the e4m3 value nearest to the rational y (ties: even code),
    saturating at 448, sign kept (y = 0 is taken as +0)."""
    table = e4m3_table_exact()
    a = abs(y)
    best = min(table, key=lambda c: (abs(table[c] - a), c & 1))
    if a >= 448:
        best = 0x7E
    return best | (0x80 if y < 0 else 0)


def fp8_pin_golden_codes(orc):
    rows = read_golden("e4m3_codes.txt")
    y = np.array([float(r[0]) for r in rows], np.float32)
    want = [int(r[1], 16) for r in rows]
    assert orc.e4m3_round(y).tolist() == want
    finite = [c for c in want if (c & 0x7F) != 0x7F]
    assert np.all(np.isfinite(orc.e4m3_value(np.array(finite, np.uint8))))
    assert orc.e4m3_value(np.array([0x7E], np.uint8))[0] == 448.0
    assert orc.e4m3_value(np.array([0x01], np.uint8))[0] == 2.0 ** -9
    assert np.isnan(orc.e4m3_value(np.array([0x7F, 0xFF], np.uint8))).all()


def fp8_pin_value_table(orc):
    table = e4m3_table_exact()
    codes = np.arange(256, dtype=np.uint8)
    v = orc.e4m3_value(codes)
    for c in range(256):
        if (c & 0x7F) == 0x7F:
            assert np.isnan(v[c])
            continue
        want = table[c & 0x7F] * (-1 if c & 0x80 else 1)
        assert Fraction(float(v[c])) == want, hex(c)
    # every finite code survives value -> code (including -0 = 0x80)
    finite = codes[(codes & 0x7F) != 0x7F]
    assert np.array_equal(orc.e4m3_round(orc.e4m3_value(finite).astype(np.float32)), finite)


def fp8_pin_rounding_exact(orc, seed=31):
    """Random fp32 values across every binade, the exact midpoints between
    neighbouring codes, and their fp32 neighbours: codes equal the nearest
    exact e4m3 value (ties even)."""
    rng = np.random.default_rng(seed)
    table = e4m3_table_exact()
    mids = [float((table[c] + table[c + 1]) / 2) for c in range(126)]
    ys = [np.float32(m) for m in mids]
    ys += [np.nextafter(np.float32(m), np.float32(np.inf)) for m in mids]
    ys += [np.nextafter(np.float32(m), np.float32(0)) for m in mids]
    ys += list((rng.standard_normal(400) * np.exp2(rng.integers(-12, 10, 400))).astype(np.float32))
    ys += [np.float32(460.0), np.float32(-1e6), np.float32(464.0)]
    y = np.array(ys, np.float32)
    y = np.concatenate([y, -y])
    got = orc.e4m3_round(y)
    for yi, gi in zip(y, got):
        assert int(gi) == e4m3_nearest_exact(Fraction(float(yi))) or (yi == 0 and int(gi) in (0, 0x80)), (yi, gi)


def fp8_pin_quantized_row_golden(orc):
    g = {r[0]: r[1:] for r in read_golden("fp8_row.txt")}
    x = np.array([float(t) for t in g["x"]], np.float32)
    bits = f32_to_bf16_bits(x)
    assert np.array_equal(bits_to_f64(bits), x.astype(np.float64))   # all exact in bf16
    c, s = orc.quantize_fp8_per_token_head(bits[None])
    assert float(s[0]) == float(g["scale"][0])
    assert c[0].tolist() == [int(t, 16) for t in g["codes"]]


def fp8_pin_quantized_rows_exact(orc, seed=32):
    """Away from ties, fp32 x / fl(a/448) rounds like the exact 448 x / a;
    the absmax element maps to +-448; the dequantised row is within half an
    e4m3 spacing of x; zero rows give s = 0 and codes 0."""
    rng = np.random.default_rng(seed)
    x = f32_to_bf16_bits(rng.standard_normal((24, 128)).astype(np.float32) * 3.0)
    x[5] = 0
    c, s = orc.quantize_fp8_per_token_head(x)
    xs = bits_to_f64(x)
    table = e4m3_table_exact()
    mids = sorted((table[i] + table[i + 1]) / 2 for i in range(126))
    checked = 0
    for r in range(x.shape[0]):
        if r == 5:
            assert s[r] == 0 and np.all(c[r] == 0)
            continue
        a = max(abs(Fraction(float(t))) for t in xs[r])
        assert float(s[r]) == float(np.float32(np.float32(a) / np.float32(448)))
        for d in range(x.shape[1]):
            exact = Fraction(448) * Fraction(float(xs[r, d])) / a
            if any(abs(abs(exact) - m_) < Fraction(1, 1 << 20) * max(m_, Fraction(1, 1 << 9)) for m_ in mids):
                continue
            assert int(c[r, d]) == e4m3_nearest_exact(exact), (r, d)
            checked += 1
        assert np.max(np.abs(orc.e4m3_value(c[r]))) == 448.0
        err = np.abs(xs[r] - orc.e4m3_value(c[r]) * float(s[r]))
        # half a spacing: 2^-4 relative for normals, 2^-10 absolute (times s) below 2^-6
        assert np.all(err <= (np.abs(xs[r]) * 2.0 ** -4 + float(s[r]) * 2.0 ** -10) * (1 + 1e-6))
    assert checked > 0.99 * (x.size - x.shape[1])


FP8_PINS = [fp8_pin_golden_codes, fp8_pin_value_table, fp8_pin_rounding_exact, fp8_pin_quantized_row_golden,
            fp8_pin_quantized_rows_exact]


@pytest.mark.parametrize("pin", FP8_PINS, ids=[p.__name__ for p in FP8_PINS])
def test_fp8_pin(pin):
    pin(oracle)


def test_e4m3_matches_torch_cast():
    """torch's float8_e4m3fn cast (round to nearest even) on every in-range
    value class: midpoints, their neighbours, random values, subnormals."""
    rng = np.random.default_rng(33)
    mags = oracle.e4m3_value(np.arange(0x7F, dtype=np.uint8))
    mids = (mags[:-1] + mags[1:]) / 2
    y = np.concatenate([mids, np.nextafter(mids.astype(np.float32), np.float32(np.inf)),
                        np.nextafter(mids.astype(np.float32), np.float32(0)), mags,
                        rng.uniform(-448, 448, 20000), rng.standard_normal(20000) * 2.0 ** -8]).astype(np.float32)
    y = np.concatenate([y, -y])
    y = y[np.abs(y) <= 448.0]
    want = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_round(y), want)


def test_fp8_store_and_gather():
    rng = np.random.default_rng(34)
    ps, T, H, D, pool = 4, 6, 2, 16, 5
    k, v = rand_bits(rng, (T, H, D)), rand_bits(rng, (T, H, D))
    v[4, 0] = 0x8000          # -0.0 everywhere: absmax 0
    slots = np.array([0, 5, 6, -1, 19, 11], np.int32)
    ck = np.zeros((pool, H, ps, D), np.uint8)
    cv = np.zeros_like(ck)
    sk = np.zeros((pool, H, ps), np.float32)
    sv = np.zeros_like(sk)
    oracle.store_fp8(ck, cv, sk, sv, k, v, slots, ps)
    assert sv[4, 0, 3] == 0 and np.all(cv[4, 0, 3] == 0)
    bt_row = np.arange(pool, dtype=np.int32)
    for t, slot in enumerate(slots):
        if slot < 0:
            continue
        p, o = divmod(int(slot), ps)
        c1, s1 = oracle.quantize_fp8_per_token_head(v[t])
        assert np.array_equal(cv[p, :, o], c1) and np.array_equal(sv[p, :, o], s1)
        for h in range(H):
            got = oracle.gather_rows(ck, sk, bt_row, [slot], h, ps)[0]
            x = bits_to_f64(k[t, h])
            assert np.all(np.abs(got - x) <= np.abs(x) * 2.0 ** -4 + sk[p, h, o] * 2.0 ** -10 + 1e-12)


def _fp8_mutants():
    import importlib.util

    def clone():
        spec = importlib.util.spec_from_file_location("oracle_fp8_mutant", oracle.__file__)
        m = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(m)
        return m

    out = {}
    m = clone()
    base_round = m.e4m3_round

    def round_ties_away(y):
        y = np.asarray(y, np.float32)
        c = base_round(y)
        # nudge exact ties away from zero
        up = base_round(np.nextafter(np.abs(y), np.float32(np.inf)) * np.sign(y))
        mags = m.e4m3_value(np.arange(0x7F, dtype=np.uint8))
        tie = np.isin(np.abs(y).astype(np.float64), (mags[:-1] + mags[1:]) / 2)
        return np.where(tie, up, c).astype(np.uint8)
    m.e4m3_round = round_ties_away
    out["ties away from zero"] = m
    m = clone()
    base_value = m.e4m3_value
    m.e4m3_value = lambda c: base_value(c) * 2.0
    out["exponent bias 6"] = m
    m = clone()
    m.E4M3_MAX = 240.0
    out["scale from the e5m2-like range"] = m
    m = clone()
    m.e4m3_round = lambda y: base_round(np.abs(np.asarray(y, np.float32)))
    out["sign dropped"] = m
    return out


@pytest.mark.parametrize("name", list(_fp8_mutants().keys()))
def test_fp8_planted_mistake_is_caught(name):
    mutant = _fp8_mutants()[name]
    failures = 0
    for pin in FP8_PINS:
        try:
            pin(mutant)
        except (AssertionError, IndexError, ValueError):
            failures += 1
    assert failures >= 1, f"no fp8 pin caught: {name}"


# ---------------------------------------------------------------------------
# layer map pins (numbers printed by the pages)
# ---------------------------------------------------------------------------

def e_series(n_layers, period, n_owning, hkv, share=True):
    layers = []
    for i in range(n_layers):
        full = (i % period) == period - 1
        src = KV_OWN if (i < n_owning or not share) else KV_AUTO
        layers.append(lay(FULL if full else SLIDING, 512 if full else 256, 8, hkv, 512, src))
    return layers


def test_kv_bytes_per_token_golden():
    models = {"E2B": (35, 5, 15, 1), "E4B": (42, 6, 24, 2)}
    # the page gives one figure for "the 8-bit formats": int8 and fp8 alike
    fmt = {"bf16": [oracle.KV_BF16], "int8": [oracle.KV_INT8, oracle.KV_FP8]}
    rows = read_golden("kv_bytes_per_token.txt")
    assert len(rows) == 8
    for model, f, sharing, full, window in rows:
        n, per, own, hkv = models[model]
        layers = e_series(n, per, own, hkv, share=(sharing == "after"))
        for kd in fmt[f]:
            assert oracle.kv_bytes_per_token(layers, FULL, kd) == int(full)
            assert oracle.kv_bytes_per_token(layers, SLIDING, kd) == int(window)


def test_slab_counts_sources_and_ratios():
    # "FreeToken PR #898", Test section: main holds 7/28 (E2B) and 7/35 (E4B) slabs
    assert oracle.slab_counts(e_series(35, 5, 15, 1, share=False)) == {FULL: 7, SLIDING: 28}
    assert oracle.slab_counts(e_series(42, 6, 24, 2, share=False)) == {FULL: 7, SLIDING: 35}
    e2b, e4b = e_series(35, 5, 15, 1), e_series(42, 6, 24, 2)
    assert oracle.slab_counts(e2b) == {FULL: 3, SLIDING: 12}
    assert oracle.slab_counts(e4b) == {FULL: 4, SLIDING: 20}
    # description, first bullet: sources 14 / 13 on E2B and 23 / 22 on E4B
    assert sorted(set(s for s in oracle.resolve_kv_sources(e2b) if s >= 0)) == [13, 14]
    assert sorted(set(s for s in oracle.resolve_kv_sources(e4b) if s >= 0)) == [22, 23]
    # shared layers hold 57% (E2B) / 43% (E4B) of the per-token KV; 7/3 and 7/4 the tokens
    for n, per, own, hkv, share_pct, ratio in [(35, 5, 15, 1, 57, Fraction(7, 3)),
                                               (42, 6, 24, 2, 43, Fraction(7, 4))]:
        before = sum(oracle.kv_bytes_per_token(e_series(n, per, own, hkv, False), k, 0) for k in (0, 1))
        after = sum(oracle.kv_bytes_per_token(e_series(n, per, own, hkv), k, 0) for k in (0, 1))
        assert Fraction(before, after) == ratio
        assert round(100 * (before - after) / before) == share_pct


def test_unsourced_shared_layer_is_refused():
    # review thread: a shared layer with no earlier layer of its type is refused
    with pytest.raises(oracle.UnsupportedLayout):
        oracle.resolve_kv_sources([lay(FULL, 512, 8, 1), lay(SLIDING, 256, 8, 1, 512, KV_AUTO)])
    with pytest.raises(oracle.UnsupportedLayout):   # a shared layer is not a source
        oracle.resolve_kv_sources([lay(FULL, 512, 8, 1), lay(FULL, 512, 8, 1, 0, KV_AUTO),
                                   lay(FULL, 512, 8, 1, 0, 1)])
    with pytest.raises(oracle.UnsupportedLayout):   # geometry must match
        oracle.resolve_kv_sources([lay(FULL, 512, 8, 1), lay(FULL, 512, 8, 2, 0, KV_AUTO)])


def test_window_matches_inclusive_window_left():
    """"pegainfer issue #807", Description: Gemma's W counts the current token,
    FlashInfer's window_left is an inclusive distance, so W maps to W - 1."""
    for W in [1, 2, 7, 1024]:
        for q in [0, 1, W - 1, W, W + 5, 3000]:
            lo, hi = oracle.visible_keys(q, SLIDING, W)
            window_left = W - 1
            keys = [k for k in range(q + 1) if q - k <= window_left]
            assert (lo, hi) == (keys[0], keys[-1])
            assert hi - lo + 1 == min(W, q + 1)


# ---------------------------------------------------------------------------
# planted mistakes: each must break at least one pin
# ---------------------------------------------------------------------------

def _mutants():
    import importlib.util

    def clone():
        # a fresh copy of the oracle module, so patched names are the ones its functions call
        spec = importlib.util.spec_from_file_location("oracle_mutant", oracle.__file__)
        m = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(m)
        return m

    out = {}
    m = clone()
    m.visible_keys = lambda q, kind, W: (0, q) if kind == FULL else (max(0, q - W), q)
    out["window off by one"] = m
    m = clone()
    m.softmax_attention = lambda q, K, V, sc: oracle.softmax_attention(q, K, V, 1.0)
    out["scale dropped"] = m
    m = clone()

    def gather_bad(slab, scales, bt, pos, h, ps):
        pos = np.asarray(pos)
        return oracle.gather_rows(slab, scales, bt, np.minimum(pos + (pos % ps == 1), pos.max()), h, ps)
    m.gather_rows = gather_bad
    out["page offset misread"] = m
    m = clone()

    def decode_swapped(layers, li, slabs, *a, **kw):
        return oracle.paged_decode(layers, li, {o: (e[1], e[0]) + tuple(e[2:]) for o, e in slabs.items()},
                                   *a, **kw)
    m.paged_decode = decode_swapped
    out["K and V swapped"] = m
    m = clone()

    def softmax_no_max(q, K, V, sc):
        s = sc * (K @ q)
        e = np.exp(s)
        return (e / e.sum()) @ V, np.log(e.sum()) + 1.0, e / e.sum()
    m.softmax_attention = softmax_no_max
    out["lse term dropped"] = m
    return out


@pytest.mark.parametrize("name", list(_mutants().keys()))
def test_planted_mistake_is_caught(name):
    mutant = _mutants()[name]
    failures = 0
    for pin in PINS:
        try:
            pin(mutant)
        except (AssertionError, IndexError, ValueError):
            failures += 1
    assert failures >= 1, f"no pin caught: {name}"
