"""Extend (chunked prefill) parity: the tcgen05 kernel through the C ABI
against the fp64 oracle.

Each case pages a seeded prefix into a permuted pool, brings a seeded chunk
of new tokens (q, k_ext, v_ext) and compares every output row (small cases)
or sampled rows (the chunked-prefill workload) with the oracle, which reads
the generator's prefix values and the same chunk.  Tolerance: max-abs 1e-2
and relative L2 2e-2 for the bf16 outputs; lse within 2e-3.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from paged_case import assert_close, bits

pytestmark = pytest.mark.gpu


class ExtendCase:
    """One extend call per layer over a paged prefix plus a chunk."""

    def __init__(self, layers, prefix, chunk, seed=0, page_size=16, device="cuda", poison_tail=True,
                 early_metadata=False, poison_window=True, split=None):
        import full_attention_gb300 as fa
        self.fa = fa
        self.layers = layers
        self.prefix = np.asarray(prefix, np.int32)
        self.chunk = np.asarray(chunk, np.int32)
        self.B = len(prefix)
        self.ps = page_size
        self.seed = seed
        self.device = device
        total = self.prefix + self.chunk
        plan = W.plan_pages(np.maximum(total, 1), page_size, seed)
        self.bt_np = plan.block_table
        self.cache = fa.Cache(layers, plan.num_pages, page_size)
        flags = (fa.FLAG_EARLY_METADATA if early_metadata else 0) | (fa.FLAG_EXTEND_SPLIT_ALL if split == "all" else 0)
        if flags:
            self.cache.set_flags(flags)
        self.ws = None
        if split is not None:
            # the split workspace: "tail" splits as the bench launches do
            # (the last wave's jobs when worth it), "all" every job it holds
            self.ws = fa.workspace(fa.extend_workspace_bytes(), device)
            self.cache.bind_extend_workspace(self.ws)
        self.src = [self.cache.source(i) for i in range(len(layers))]
        self.slabs = self.cache.allocate(device)
        for i, (k, v, _, _) in self.slabs.items():
            k.copy_(W.randn_bf16(tuple(k.shape), seed * 100 + 10 + 2 * i, device))
            v.copy_(W.randn_bf16(tuple(v.shape), seed * 100 + 11 + 2 * i, device))
            if poison_tail:
                self._poison(k, v)
            if poison_window:
                self._poison_before_window(i, k, v)
        self.indptr = np.concatenate([[0], np.cumsum(self.chunk)]).astype(np.int32)
        self.N = int(self.indptr[-1])
        self.q, self.kx, self.vx = {}, {}, {}
        for i, d in enumerate(layers):
            self.q[i] = W.randn_bf16((max(self.N, 1), d["num_q_heads"], d["head_dim"]), seed * 100 + 20 + 3 * i, device)
        for i, d in enumerate(layers):
            if self.src[i] == i:
                self.kx[i] = W.randn_bf16((max(self.N, 1), d["num_kv_heads"], d["head_dim"]), seed * 100 + 21 + 3 * i,
                                          device)
                self.vx[i] = W.randn_bf16((max(self.N, 1), d["num_kv_heads"], d["head_dim"]), seed * 100 + 22 + 3 * i,
                                          device)
        self.bt = torch.from_numpy(self.bt_np).to(device)
        self.indptr_dev = torch.from_numpy(self.indptr).to(device)
        self.prefix_dev = torch.from_numpy(self.prefix).to(device)
        torch.cuda.synchronize()

    def _poison(self, k, v):
        """NaN every slot at or past a sequence's prefix: extend must read only
        positions < P from the slab (the chunk comes from k_ext / v_ext)."""
        mask = torch.zeros(k.shape[0], self.ps, dtype=torch.bool)
        for b in range(self.B):
            for pos in range(int(self.prefix[b]), int(self.prefix[b] + self.chunk[b])):
                mask[self.bt_np[b, pos // self.ps], pos % self.ps] = True
        mask = mask.to(self.device)[:, None, :, None].expand_as(k)
        k.masked_fill_(mask, float("nan"))
        v.masked_fill_(mask, float("nan"))

    def _poison_before_window(self, o, k, v):
        """NaN the slots of a sliding slab before every query's window: the
        first query of sequence b sits at P_b and sees keys > P_b - W.  The
        page holding P_b - W + 1 is read from its 16-row boundary, so this
        puts NaN inside a tile the kernel copies."""
        ws = [d["window"] for j, d in enumerate(self.layers) if self.src[j] == o and d["kind"] == W.SLIDING]
        if not ws:
            return
        mask = torch.zeros(k.shape[0], self.ps, dtype=torch.bool)
        for b in range(self.B):
            for pos in range(0, max(0, int(self.prefix[b]) - max(ws) + 1)):
                mask[self.bt_np[b, pos // self.ps], pos % self.ps] = True
        mask = mask.to(self.device)[:, None, :, None].expand_as(k)
        k.masked_fill_(mask, float("nan"))
        v.masked_fill_(mask, float("nan"))

    def run(self, i, out=None, lse=None):
        d = self.layers[i]
        o = self.src[i]
        if out is None:
            out = torch.full((max(self.N, 1), d["num_q_heads"], d["head_dim"]), float("nan"), dtype=torch.bfloat16,
                             device=self.device)
        if lse is None:
            lse = torch.full((max(self.N, 1), d["num_q_heads"]), float("nan"), dtype=torch.float32,
                             device=self.device)
        self.cache.extend(i, self.q[i][: self.N], self.kx[o][: self.N], self.vx[o][: self.N], self.indptr_dev,
                          self.prefix_dev, self.bt, int(self.chunk.max()), int(max(self.prefix.max(), 0)), out, lse)
        self.lse = lse
        return out[: self.N]

    def oracle(self, i, rows=None):
        """Oracle out [N][Hq][D] (optionally only `rows` (token, head) pairs)."""
        o = self.src[i]
        k, v, _, _ = self.slabs[o]
        # the generator's values (the poison touches only slots the oracle never reads)
        sk = bits(W.randn_bf16(tuple(k.shape), self.seed * 100 + 10 + 2 * o, self.device))
        sv = bits(W.randn_bf16(tuple(v.shape), self.seed * 100 + 11 + 2 * o, self.device))
        out, lse = oracle.paged_extend(self.layers, i, {o: (sk, sv)}, bits(self.q[i][: self.N]),
                                       bits(self.kx[o][: self.N]), bits(self.vx[o][: self.N]), self.indptr,
                                       self.prefix, self.bt_np, self.ps, rows=rows)
        self.oracle_lse = lse
        return out


def lay(kind, D, hq, hkv, Wn=0, src=W.KV_OWN):
    return W.layer(kind, D, hq, hkv, Wn, src)


SMALL = [
    # (layer, prefix, chunk)
    (lay(W.SLIDING, 256, 4, 2, 48), [40, 0, 100, 17], [37, 20, 130, 1]),
    (lay(W.FULL, 512, 8, 1), [40, 0, 100, 17], [37, 20, 130, 1]),
    (lay(W.FULL, 256, 16, 8), [64, 3], [64, 200]),
    (lay(W.SLIDING, 512, 16, 2, 100), [300, 33], [90, 160]),
    (lay(W.FULL, 256, 2, 2), [0, 129], [257, 64]),
    (lay(W.SLIDING, 256, 8, 1, 1), [20, 0], [45, 16]),
]


@pytest.mark.parametrize("spec", SMALL, ids=[f"{'F' if s[0]['kind'] == 0 else 'S'}{s[0]['head_dim']}"
                                             f"_g{s[0]['num_q_heads'] // s[0]['num_kv_heads']}_W{s[0]['window']}"
                                             for s in SMALL])
def test_small_extend(spec):
    layer, prefix, chunk = spec
    c = ExtendCase([layer], prefix, chunk, seed=7)
    out = c.run(0)
    ref = c.oracle(0)
    assert_close(out, ref, what="extend")
    g = c.lse[: c.N].double().cpu().numpy()
    assert np.all(np.abs(g - c.oracle_lse) <= 2e-3 * np.maximum(1.0, np.abs(c.oracle_lse)))
    assert c.fa.device_error() == 0


@pytest.mark.parametrize("spec", SMALL, ids=[f"{'F' if s[0]['kind'] == 0 else 'S'}{s[0]['head_dim']}"
                                             f"_g{s[0]['num_q_heads'] // s[0]['num_kv_heads']}_W{s[0]['window']}"
                                             for s in SMALL])
def test_small_extend_split(spec):
    """Every job split over two CTAs (the first and second half of its key
    tiles) and merged through the workspace: the same parity with the
    oracle, and the workspace's arrival counters are zero afterwards."""
    layer, prefix, chunk = spec
    c = ExtendCase([layer], prefix, chunk, seed=7, split="all")
    out = c.run(0)
    assert_close(out, c.oracle(0), what="split extend")
    g = c.lse[: c.N].double().cpu().numpy()
    assert np.all(np.abs(g - c.oracle_lse) <= 2e-3 * np.maximum(1.0, np.abs(c.oracle_lse)))
    assert c.fa.device_error() == 0
    cap = (torch.cuda.get_device_properties(0).multi_processor_count // 2) or 1
    assert int(c.ws[: 4 * cap].view(torch.int32).abs().sum()) == 0
    # a second call over the same workspace gives the same output
    assert torch.equal(c.run(0), out)


def test_split_workspace_for_one_job_and_unbinding():
    """A workspace with room for one job's partials splits only the last job of
    the launch (the rest run whole); the output still matches the oracle.
    Unbinding returns to the unsplit kernel, bit for bit the same as a cache
    that never had a workspace."""
    layer = lay(W.FULL, 512, 8, 1)
    c = ExtendCase([layer], [40, 100, 17], [37, 130, 1], seed=11, split="all")
    one = 256 + 4096 + 2 * 128 * 256 * 4   # counters, 128 rows x 16 B x 2 CTAs, 2 partials of 128 x 256 fp32
    small = c.fa.workspace(one)
    c.cache.bind_extend_workspace(small)
    assert_close(c.run(0), c.oracle(0), what="one split job")
    assert c.fa.device_error() == 0
    assert int(small[:4].view(torch.int32).abs().sum()) == 0
    c.cache.bind_extend_workspace(None)
    unsplit = c.run(0).clone()
    plain = ExtendCase([layer], [40, 100, 17], [37, 130, 1], seed=11)
    assert torch.equal(unsplit, plain.run(0))
    with pytest.raises(c.fa.FAError):
        c.cache.bind_extend_workspace(c.fa.workspace(one - 256))   # too small for one job


@pytest.mark.parametrize("split", [None, "all"])
def test_length_past_its_bound_sets_error_bit(split):
    """A prefix longer than max_prefix_len, or a chunk longer than max_q_len,
    is cut to the bound and reported with FA_DEV_ERR_BOUND (several row blocks
    per sequence: g = 2 packs 64 tokens per block)."""
    layer = lay(W.FULL, 256, 4, 2)
    c = ExtendCase([layer], [40, 300], [150, 200], seed=10, split=split)
    d = c.layers[0]
    out = torch.zeros((c.N, d["num_q_heads"], d["head_dim"]), dtype=torch.bfloat16, device="cuda")
    assert c.fa.device_error() == 0
    # prefix 300 against a bound of 256
    c.cache.extend(0, c.q[0][: c.N], c.kx[0][: c.N], c.vx[0][: c.N], c.indptr_dev, c.prefix_dev, c.bt, 200, 256, out)
    assert c.fa.device_error() & c.fa.DEV_ERR_BOUND
    # chunk 200 against a bound of 128 (the launch covers 128 tokens per sequence)
    c.cache.extend(0, c.q[0][: c.N], c.kx[0][: c.N], c.vx[0][: c.N], c.indptr_dev, c.prefix_dev, c.bt, 128, 300, out)
    assert c.fa.device_error() & c.fa.DEV_ERR_BOUND
    # within both bounds: no bit
    c.cache.extend(0, c.q[0][: c.N], c.kx[0][: c.N], c.vx[0][: c.N], c.indptr_dev, c.prefix_dev, c.bt, 200, 300, out)
    assert c.fa.device_error() == 0


def test_shared_layer_extend_reads_source_slab_and_chunk():
    layers = [lay(W.SLIDING, 256, 8, 2, 64), lay(W.FULL, 512, 8, 1), lay(W.SLIDING, 256, 8, 2, 64, W.KV_AUTO)]
    c = ExtendCase(layers, [50, 130], [70, 20], seed=8)
    assert c.src == [0, 1, 0]
    a = c.run(2)
    assert_close(a, c.oracle(2), what="shared extend")
    # the shared layer with the source's q equals the source layer
    c.q[2] = c.q[0]
    assert torch.equal(c.run(2), c.run(0))


def test_extend_equals_decode_at_the_last_position_and_early_metadata():
    layer = lay(W.FULL, 512, 8, 1)
    c = ExtendCase([layer], [77], [40], seed=9)
    out = c.run(0)
    e = ExtendCase([layer], [77], [40], seed=9, early_metadata=True)
    assert torch.equal(out, e.run(0))
    # decode of the last chunk token after storing the chunk equals extend's last row
    slots = W.slots_for_positions(c.bt_np[0], np.arange(77, 117), 16)
    c.cache.store(0, c.kx[0][:40], c.vx[0][:40], torch.from_numpy(slots).cuda())
    dq = c.q[0][39:40].contiguous()
    dout = torch.empty_like(dq)
    ws = c.fa.workspace(c.cache.decode_workspace_bytes(0, 1, 117))
    c.cache.decode(0, dq, c.bt[:1], torch.tensor([117], dtype=torch.int32, device="cuda"), 117, dout, None, ws)
    assert_close(dout[0], out[39].double().cpu().numpy(), atol=1e-2, rel=2e-2, what="decode vs extend")


@pytest.mark.parametrize("split", [None, "tail"])
def test_chunked_prefill_workload(split):
    """The chunked-prefill workload: 4 prompts of 4096 tokens in 512-token
    chunks.  Chunks 0, 3 and 7 of both layers are compared on sampled rows,
    without and with the split workspace the bench binds (its head_dim-512
    launches of 512 jobs then split their last wave on a 152-SM device)."""
    w = W.chunked_prefill()
    B, S, Cn = w.batch, w.prompt_len, w.chunk
    rng = np.random.default_rng(2)
    for ci in (0, 3, 7):
        P = ci * Cn
        c = ExtendCase(w.layers, [P] * B, [Cn] * B, seed=20 + ci, split=split)
        for li in range(2):
            out = c.run(li)
            d = w.layers[li]
            toks = sorted(set(rng.choice(c.N, size=24, replace=False).tolist() + [0, c.N - 1, Cn - 1, Cn]))
            rows = [(t, j) for t in toks for j in range(d["num_q_heads"])]
            ref = c.oracle(li, rows=rows)
            idx = torch.tensor(toks)
            assert_close(out[idx], ref[toks], what=f"chunk {ci} layer {li}")
        assert c.fa.device_error() == 0


def test_large_scores_keep_parity_and_report_out_of_range():
    """A chunk key of 65280 makes its scores reach thousands (log2 units): the
    two softmax halves of a row still agree on an exact base and the result
    matches the oracle.  A score past the 16-bit base range (a q element and
    a key element of 60000) is reported as FA_DEV_ERR_RANGE."""
    for layer in (lay(W.SLIDING, 256, 8, 2, 64), lay(W.FULL, 512, 8, 1)):
        c = ExtendCase([layer], [40, 100], [37, 130], seed=11)
        c.kx[0][5, 0, 3] = 65280.0
        out = c.run(0)
        assert_close(out, c.oracle(0), what="large key")
        assert c.fa.device_error() == 0
        c.q[0][20, 0, 3] = 60000.0
        c.kx[0][5, 0, 3] = 60000.0
        c.run(0)
        assert c.fa.device_error() == c.fa.DEV_ERR_RANGE
