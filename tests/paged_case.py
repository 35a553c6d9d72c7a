"""Builds seeded decode cases on the GPU and the matching oracle inputs.

Inputs come only from the seeded generators (workloads.py).  The oracle never
reads a value that a library kernel wrote: its slabs are the generator's
bf16 values, updated by the oracle's own store (bf16 copy or int8
quantisation) of the same new rows the GPU store receives.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads as W

ATOL, RTOL = 1e-2, 2e-2   # max-abs and relative-L2 bounds for bf16 outputs


def assert_close(got, ref, atol=ATOL, rel=RTOL, what=""):
    g = got.detach().double().cpu().numpy() if torch.is_tensor(got) else np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = float(np.max(np.abs(g - ref))) if g.size else 0.0
    nrm = float(np.linalg.norm(ref))
    relv = float(np.linalg.norm(g - ref)) / nrm if nrm > 0 else float(np.linalg.norm(g - ref))
    assert err <= atol and relv <= rel, f"{what}: max-abs {err:.3e} (<= {atol}), rel-L2 {relv:.3e} (<= {rel})"
    return err, relv


def bits(t):
    return W.bf16_bits(t)


class DecodeCase:
    """One decode step of a layer stack: slabs filled with seeded context, the
    current token's k, v stored through the library, then attention per layer."""

    def __init__(self, layers, lens, page_size=16, kv_dtype=W.KV_BF16, seed=0, device="cuda",
                 window_table=False, poison=False, pool_factor=1.25, min_pool=0, window_pool=False):
        import full_attention_gb300 as fa
        self.fa = fa
        self.layers = layers
        self.lens = np.asarray(lens, np.int32)
        self.B = len(lens)
        self.ps = page_size
        self.kv_dtype = kv_dtype
        self.seed = seed
        self.device = device
        self.max_len = int(self.lens.max())
        self.poison = poison
        full = W.plan_pages(self.lens, page_size, seed, pool_factor, min_pool)
        self.plans = {}
        num_pages = full.num_pages
        for i, d in enumerate(layers):
            if d["kind"] == W.SLIDING and window_table:
                plan = W.plan_pages(self.lens, page_size, seed + 1000, pool_factor, min_pool, window=d["window"],
                                    max_pages=full.block_table.shape[1])
            else:
                plan = full
            self.plans[i] = plan
            num_pages = max(num_pages, plan.num_pages)
        self.num_pages = num_pages
        if window_pool:
            # the sliding layers' tables (in-window pages only) index a pool of their own
            assert window_table
            full_pages = [self.plans[i].num_pages for i, d in enumerate(layers) if d["kind"] == W.FULL]
            win_pages = [self.plans[i].num_pages for i, d in enumerate(layers) if d["kind"] == W.SLIDING]
            self.num_pages = max(full_pages or [full.num_pages])
            self.window_pages = max(win_pages)
        self.cache = fa.Cache(layers, self.num_pages, page_size, kv_dtype)
        if window_pool:
            self.cache.set_window_pool(self.window_pages)
        self.src = [self.cache.source(i) for i in range(len(layers))]
        self.slabs = self.cache.allocate(device)
        self.bt_dev = {i: torch.from_numpy(self.plans[i].block_table).to(device) for i in range(len(layers))}
        self.lens_dev = torch.from_numpy(self.lens).to(device)
        self.q = {}
        self.new_kv = {}
        self._ctx_rows = {}
        for i, d in enumerate(layers):
            self.q[i] = W.randn_bf16((self.B, d["num_q_heads"], d["head_dim"]), seed * 100 + 3 * i + 1, device)
        for i, d in enumerate(layers):
            if self.src[i] != i:
                continue
            self._fill_context(i, d)
            k = W.randn_bf16((self.B, d["num_kv_heads"], d["head_dim"]), seed * 100 + 3 * i + 2, device)
            v = W.randn_bf16((self.B, d["num_kv_heads"], d["head_dim"]), seed * 100 + 3 * i + 3, device)
            self.new_kv[i] = (k, v)
        torch.cuda.synchronize()

    # -- context ------------------------------------------------------------
    def _visible_lo(self, d, L):
        return max(0, L - d["window"]) if d["kind"] == W.SLIDING else 0

    def _fill_context(self, i, d):
        k_s, v_s, ks_s, vs_s = self.slabs[i]
        shape = tuple(k_s.shape)
        if self.kv_dtype == W.KV_BF16:
            k_s.copy_(W.randn_bf16(shape, self.seed * 100 + 50 + 2 * i, self.device))
            v_s.copy_(W.randn_bf16(shape, self.seed * 100 + 51 + 2 * i, self.device))
            if self.poison:
                self._poison(i, d)
            return
        # 8-bit: quantise seeded bf16 context rows through the library's store;
        # slots it does not write keep junk codes (e4m3: the NaN codes)
        nan = torch.tensor(float("nan"))
        k_s.fill_(0x7F if self.kv_dtype == W.KV_FP8 else 77)
        v_s.fill_(0xFF if self.kv_dtype == W.KV_FP8 else -77)
        ks_s.fill_(nan)
        vs_s.fill_(nan)
        rows, slots = [], []
        for b, L in enumerate(self.lens):
            lo = self._visible_lo(d, int(L))
            pos = np.arange(lo, int(L) - 1)
            rows.append((b, lo, int(L) - 1))
            slots.append(W.slots_for_positions(self.plans[i].block_table[b], pos, self.ps))
        slot = torch.from_numpy(np.concatenate(slots)).to(self.device)
        T = int(slot.numel())
        k = W.randn_bf16((T, d["num_kv_heads"], d["head_dim"]), self.seed * 100 + 60 + 2 * i, self.device)
        v = W.randn_bf16((T, d["num_kv_heads"], d["head_dim"]), self.seed * 100 + 61 + 2 * i, self.device)
        if T:
            self.cache.store(i, k, v, slot)
        self._ctx_rows[i] = (k, v, rows)

    def _poison(self, i, d):
        """NaN every slab position a query of this layer must not read."""
        k_s, v_s, _, _ = self.slabs[i]
        bt = self.plans[i].block_table
        mask = torch.ones(k_s.shape[0], self.ps, dtype=torch.bool)
        for b, L in enumerate(self.lens):
            lo = self._visible_lo(d, int(L))
            for pos in range(lo, int(L)):
                mask[bt[b, pos // self.ps], pos % self.ps] = False
        mask = mask.to(self.device)[:, None, :, None].expand_as(k_s)
        k_s.masked_fill_(mask, float("nan"))
        v_s.masked_fill_(mask, float("nan"))

    # -- the step -----------------------------------------------------------
    def slot_mapping(self, i):
        return torch.from_numpy(W.decode_slot_mapping(self.lens, self.plans[i].block_table, self.ps)).to(self.device)

    def store_current(self):
        for i, (k, v) in self.new_kv.items():
            self.cache.store(i, k, v, self.slot_mapping(i))

    def workspace(self, i):
        n = self.cache.decode_workspace_bytes(i, self.B, self.max_len)
        return self.fa.workspace(n, self.device) if n else None

    def decode(self, i, out=None, lse=None, ws=None):
        d = self.layers[i]
        if out is None:
            out = torch.empty((self.B, d["num_q_heads"], d["head_dim"]), dtype=torch.bfloat16, device=self.device)
        if lse is None:
            lse = torch.empty((self.B, d["num_q_heads"]), dtype=torch.float32, device=self.device)
        if ws is None:
            ws = self.workspace(i)
        self.cache.decode(i, self.q[i], self.bt_dev[i], self.lens_dev, self.max_len, out, lse, ws)
        return out, lse

    def decode_store(self, i, out=None, lse=None, ws=None, slots=None):
        """The fused call: store layer i's current rows (owning layer) and decode."""
        d = self.layers[i]
        if out is None:
            out = torch.empty((self.B, d["num_q_heads"], d["head_dim"]), dtype=torch.bfloat16, device=self.device)
        if lse is None:
            lse = torch.empty((self.B, d["num_q_heads"]), dtype=torch.float32, device=self.device)
        if ws is None:
            ws = self.workspace(i)
        if self.src[i] == i:
            k, v = self.new_kv[i]
            sl = self.slot_mapping(i) if slots is None else slots
        else:
            k = v = sl = None
        self.cache.decode_store(i, self.q[i], k, v, sl, self.bt_dev[i], self.lens_dev, self.max_len, out, lse, ws)
        return out, lse

    # -- oracle -------------------------------------------------------------
    def oracle_decode(self, i, seqs):
        """Oracle outputs of layer i for the sequences `seqs` (all heads),
        over compact host copies of just those sequences' pages."""
        d = self.layers[i]
        o = self.src[i]
        plan = self.plans[i]
        seqs = list(seqs)
        bt_c = np.full((len(seqs), plan.block_table.shape[1]), -1, np.int32)
        phys = []
        for n, b in enumerate(seqs):
            L = int(self.lens[b])
            lo = self._visible_lo(d, L)
            for lp in range(lo // self.ps, (L - 1) // self.ps + 1):
                bt_c[n, lp] = len(phys)
                phys.append(int(plan.block_table[b, lp]))
        idx = torch.tensor(phys, dtype=torch.long, device=self.device)
        owner_d = self.layers[o]
        if self.kv_dtype == W.KV_BF16:
            k_s, v_s, _, _ = self.slabs[o]
            # the generator's context values, before this step's store
            sk = bits(W.randn_bf16(tuple(k_s.shape), self.seed * 100 + 50 + 2 * o, self.device)[idx])
            sv = bits(W.randn_bf16(tuple(v_s.shape), self.seed * 100 + 51 + 2 * o, self.device)[idx])
            if self.poison:
                # poisoned positions are never visible; keep the oracle slab finite
                pass
            k_new, v_new = self.new_kv[o]
            slots = [bt_c[n, (int(self.lens[b]) - 1) // self.ps] * self.ps + (int(self.lens[b]) - 1) % self.ps
                     for n, b in enumerate(seqs)]
            oracle.store_bf16(sk, sv, bits(k_new[seqs]), bits(v_new[seqs]), slots, self.ps)
            slabs = {o: (sk, sv)}
        else:
            H, D = owner_d["num_kv_heads"], owner_d["head_dim"]
            store_q = oracle.store_fp8 if self.kv_dtype == W.KV_FP8 else oracle.store_int8
            ck = np.zeros((len(phys), H, self.ps, D), np.uint8 if self.kv_dtype == W.KV_FP8 else np.int8)
            cv = np.zeros_like(ck)
            sk = np.zeros((len(phys), H, self.ps), np.float32)
            sv = np.zeros_like(sk)
            k_rows, v_rows, ranges = self._ctx_rows[o]
            start = 0
            offs = {}
            for (b, lo, hi) in ranges:
                offs[b] = (start, lo, hi)
                start += hi - lo
            for n, b in enumerate(seqs):
                st, lo, hi = offs[b]
                pos = np.arange(lo, hi)
                # rows this layer's queries can see: [visible lo, L-1)
                vis_lo = self._visible_lo(d, int(self.lens[b]))
                sel = pos >= vis_lo
                kr = bits(k_rows[st:st + (hi - lo)])[sel]
                vr = bits(v_rows[st:st + (hi - lo)])[sel]
                sl = W.slots_for_positions(bt_c[n], pos[sel], self.ps)
                store_q(ck, cv, sk, sv, kr, vr, sl, self.ps)
            k_new, v_new = self.new_kv[o]
            slots = [bt_c[n, (int(self.lens[b]) - 1) // self.ps] * self.ps + (int(self.lens[b]) - 1) % self.ps
                     for n, b in enumerate(seqs)]
            store_q(ck, cv, sk, sv, bits(k_new[seqs]), bits(v_new[seqs]), slots, self.ps)
            slabs = {o: (ck, cv, sk, sv)}
        q = bits(self.q[i][seqs])
        sub_layers = [dict(l) for l in self.layers]
        out, lse = oracle.paged_decode(sub_layers, i, slabs, q, bt_c, self.lens[seqs], self.ps)
        return out, lse
