"""C-ABI checks that need no GPU: the library builds, loads, exports every
function include/fa.h declares, and its host-side logic (layer -> slab map,
source rule, refusals, bytes per token, workspace sizing) agrees with the
oracle and with the numbers the pages print."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from oracle import FULL, SLIDING, KV_AUTO, KV_OWN

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def fa():
    import __graft_entry__
    __graft_entry__.build()
    import full_attention_gb300 as fa
    return fa


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^FA_API\s+[\w\s\*]+?\b(fa_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ["fa_cache_create", "fa_cache_destroy", "fa_cache_bind_slab", "fa_cache_layer_source",
                     "fa_kv_bytes_per_token", "fa_kv_store", "fa_decode_workspace_bytes",
                     "fa_paged_decode_attn", "fa_paged_extend_attn", "fa_get_device_error", "fa_last_error"]:
        assert required in names


def test_library_exports_every_declared_symbol(fa):
    lib = ctypes.CDLL(fa.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert fa.lib().fa_version() >= 100


def lay(kind, D, hq, hkv, W=0, src=KV_OWN):
    return dict(kind=kind, head_dim=D, num_q_heads=hq, num_kv_heads=hkv, window=W if kind == SLIDING else 0,
                kv_source=src, sm_scale=float(np.float32(1 / np.sqrt(D))))


def e_series(n_layers, period, n_owning, hkv, share=True):
    out = []
    for i in range(n_layers):
        full = (i % period) == period - 1
        src = KV_OWN if (i < n_owning or not share) else KV_AUTO
        out.append(lay(FULL if full else SLIDING, 512 if full else 256, 8, hkv, 512, src))
    return out


@pytest.mark.parametrize("model", [(35, 5, 15, 1), (42, 6, 24, 2)], ids=["E2B", "E4B"])
def test_sources_and_bytes_match_oracle(fa, model):
    for share in (True, False):
        layers = e_series(*model, share=share)
        for dtype in (fa.KV_BF16, fa.KV_INT8, fa.KV_FP8):
            c = fa.Cache(layers, 64, 16, dtype)
            want = oracle.resolve_kv_sources(layers)
            got = [c.source(i) for i in range(len(layers))]
            assert got == [i if s == -1 else s for i, s in enumerate(want)]
            for kind in (FULL, SLIDING):
                assert c.bytes_per_token(kind) == oracle.kv_bytes_per_token(layers, kind, dtype)
            for i in range(len(layers)):
                kv, sc = c.slab_bytes(i)
                if want[i] == -1:
                    elem = 2 if dtype == fa.KV_BF16 else 1
                    assert kv == 64 * layers[i]["num_kv_heads"] * 16 * layers[i]["head_dim"] * elem
                    assert sc == (0 if dtype == fa.KV_BF16 else 64 * layers[i]["num_kv_heads"] * 16 * 4)
                else:
                    assert (kv, sc) == (0, 0)


def test_bytes_per_token_golden(fa):
    """The unit_bytes the "FreeToken PR #898" End-to-end section prints."""
    rows = [l.split() for l in open(os.path.join(ROOT, "tests", "golden", "kv_bytes_per_token.txt"))
            if l.strip() and not l.startswith("#")]
    models = {"E2B": (35, 5, 15, 1), "E4B": (42, 6, 24, 2)}
    for model, f, sharing, full, window in rows:
        # the page's 8-bit figures hold for the int8 and the fp8 format alike
        for dtype in ((fa.KV_INT8, fa.KV_FP8) if f == "int8" else (fa.KV_BF16,)):
            c = fa.Cache(e_series(*models[model], share=sharing == "after"), 8, 16, dtype)
            assert (c.bytes_per_token(FULL), c.bytes_per_token(SLIDING)) == (int(full), int(window))


def test_refusals(fa):
    bad_layouts = [
        [lay(FULL, 512, 8, 1), lay(SLIDING, 256, 8, 1, 512, KV_AUTO)],           # no earlier sliding owner
        [lay(FULL, 512, 8, 1), lay(FULL, 512, 8, 1, 0, KV_AUTO), lay(FULL, 512, 8, 1, 0, 1)],  # shared source
        [lay(FULL, 512, 8, 1), lay(FULL, 512, 8, 2, 0, KV_AUTO)],                # geometry differs
        [lay(SLIDING, 256, 8, 1, 512), lay(FULL, 512, 8, 1, 0, 0)],              # source of another kind
        [lay(FULL, 128, 8, 1)],                                                  # head_dim not instantiated
    ]
    for layers in bad_layouts:
        with pytest.raises(fa.FAError) as e:
            fa.Cache(layers, 8, 16)
        assert e.value.status == fa.ERR_UNSUPPORTED
    for layers, st in [([lay(SLIDING, 256, 8, 1, 0)], fa.ERR_INVALID_ARG),      # W < 1
                       ([lay(FULL, 512, 6, 4)], fa.ERR_INVALID_ARG)]:            # Hq not a multiple of Hkv
        with pytest.raises(fa.FAError) as e:
            fa.Cache(layers, 8, 16)
        assert e.value.status == st
    for ps in (8, 24, 512):
        with pytest.raises(fa.FAError) as e:
            fa.Cache([lay(FULL, 512, 8, 1)], 8, ps)
        assert e.value.status == fa.ERR_UNSUPPORTED


def test_unbound_and_shared_bind_errors(fa):
    c = fa.Cache([lay(SLIDING, 256, 8, 1, 64), lay(SLIDING, 256, 8, 1, 64, KV_AUTO)], 8, 16)
    # a shared layer cannot be bound; its source's slab is the one it reads
    with pytest.raises(fa.FAError) as e:
        c.bind(1, None, None)
    assert e.value.status == fa.ERR_INVALID_ARG
    # the store on a shared layer is a no-op that needs nothing bound
    st = fa.lib().fa_kv_store(c._h, 1, None, None, None, 4, None)
    assert st == fa.OK
    # the owner has no slab yet
    st = fa.lib().fa_kv_store(c._h, 0, None, None, None, 4, None)
    assert st == fa.ERR_NOT_BOUND


def test_decode_workspace_sizing(fa):
    for D, kind, W in [(512, FULL, 0), (256, SLIDING, 512), (256, SLIDING, 1024)]:
        c = fa.Cache([lay(kind, D, 8, 1, W)], 1024, 16)
        for B, maxlen in [(1, 200), (64, 4096), (8, 131072), (128, 8192)]:
            ws = c.decode_workspace_bytes(0, B, maxlen)
            assert ws % 4 == 0
            if ws:
                # partial outputs plus (max, sum) per split: a multiple of one row per (b, head)
                rows = B * 8
                per_split = D * 4 + 8
                assert (ws - 256) <= rows * per_split * ((maxlen + 15) // 16) + 256
    assert c.decode_workspace_bytes(0, 0, 100) == 0


def test_cache_flags(fa):
    c = fa.Cache([lay(FULL, 512, 8, 1)], 8, 16)
    c.set_flags(fa.FLAG_EARLY_METADATA)
    c.set_flags(0)
    with pytest.raises(fa.FAError) as e:
        c.set_flags(0x80)
    assert e.value.status == fa.ERR_INVALID_ARG


def test_extend_split_workspace_binding(fa):
    """The extend split workspace: its size follows the layout (arrival
    counters, per job and CTA 128 rows of 16 bytes and a 128 x 256 fp32
    partial, each part 256-byte aligned) for half the SMs' jobs; binding
    refuses a misaligned or too small buffer before any CUDA call; NULL
    unbinds; the split-every-job flag is accepted."""
    lib = ctypes.CDLL(fa.LIB_PATH)
    lib.fa_extend_workspace_bytes.restype = ctypes.c_size_t
    lib.fa_cache_bind_extend_workspace.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t]
    up = lambda b: (b + 255) // 256 * 256
    one = up(4) + up(2 * 128 * 16) + 2 * 128 * 256 * 4
    total = fa.extend_workspace_bytes()
    caps = [n for n in range(1, 2048) if up(4 * n) + up(n * 2 * 128 * 16) + n * 2 * 128 * 256 * 4 == total]
    assert len(caps) == 1 and caps[0] >= 1          # half the SM count (152 SMs: 76 jobs, about 20 MB)
    c = fa.Cache([lay(FULL, 512, 8, 1)], 8, 16)
    assert lib.fa_cache_bind_extend_workspace(c._h, 0x1000 + 16, total) == fa.ERR_INVALID_ARG
    assert lib.fa_cache_bind_extend_workspace(c._h, 0x1000, one - 1) == fa.ERR_WORKSPACE
    assert lib.fa_cache_bind_extend_workspace(c._h, None, 0) == fa.OK
    assert lib.fa_cache_bind_extend_workspace(None, None, 0) == fa.ERR_INVALID_ARG
    c.set_flags(fa.FLAG_EARLY_METADATA | fa.FLAG_EXTEND_SPLIT_ALL)
    c.set_flags(0)


def test_8bit_formats_reach_extend_and_multi_token_decode(fa):
    """Extend and multi-token decode serve the 8-bit formats: with no slab
    bound the calls stop at that check (before any pointer is read or any
    launch is made), not at a format refusal."""
    for dtype in (fa.KV_BF16, fa.KV_INT8, fa.KV_FP8):
        c = fa.Cache([lay(FULL, 512, 8, 1)], 8, 16, dtype)
        st = fa.lib().fa_paged_extend_attn(c._h, 0, None, None, None, None, None, None, 1, 2, 4, 2, 16, None, None,
                                           None)
        assert st == fa.ERR_NOT_BOUND
        st = fa.lib().fa_paged_decode_multi_attn(c._h, 0, None, None, None, None, 1, 2, 4, 2, 16, None, None, None)
        assert st == fa.ERR_NOT_BOUND


def test_window_pool_sizes_the_sliding_slabs(fa):
    """Sliding layers' slabs take the window pool's page count, full layers keep
    the cache's; a shared layer owns nothing; the per-token cost is unchanged;
    0 restores the single pool; bad sizes are refused (no GPU needed)."""
    layers = [lay(SLIDING, 256, 8, 2, 64), lay(FULL, 512, 8, 1), lay(SLIDING, 256, 8, 2, 64, KV_AUTO)]
    for dtype in (fa.KV_BF16, fa.KV_INT8, fa.KV_FP8):
        c = fa.Cache(layers, 1000, 16, dtype)
        elem = 2 if dtype == fa.KV_BF16 else 1
        per_token = (c.bytes_per_token(FULL), c.bytes_per_token(SLIDING))
        c.set_window_pool(40)
        kv, sc = c.slab_bytes(0)
        assert kv == 40 * 2 * 16 * 256 * elem and sc == (0 if dtype == fa.KV_BF16 else 40 * 2 * 16 * 4)
        assert c.slab_bytes(1)[0] == 1000 * 1 * 16 * 512 * elem
        assert c.slab_bytes(2) == (0, 0)
        assert (c.layer_pages(0), c.layer_pages(1), c.layer_pages(2)) == (40, 1000, 40)
        assert (c.bytes_per_token(FULL), c.bytes_per_token(SLIDING)) == per_token
        c.set_window_pool(0)
        assert c.slab_bytes(0)[0] == 1000 * 2 * 16 * 256 * elem
    c = fa.Cache(layers, 1000, 16)
    with pytest.raises(fa.FAError) as e:
        c.set_window_pool(-1)
    assert e.value.status == fa.ERR_INVALID_ARG
    with pytest.raises(fa.FAError) as e:
        c.set_window_pool(1 << 27)   # 2^27 pages x 2 heads x 16 rows >= 2^31
    assert e.value.status == fa.ERR_UNSUPPORTED


def test_multi_layer_decode_argument_checks(fa):
    """fa_paged_decode_attn_layers validates on the host, before any device
    access: the layer count, duplicates, one head_dim per call, pointers,
    alignment and the workspace size.  Host buffers stand in for device
    pointers (never dereferenced by the checks)."""
    import ctypes
    layers = [lay(SLIDING, 256, 8, 1, 64), lay(SLIDING, 256, 8, 1, 64), lay(FULL, 512, 8, 1)]
    c = fa.Cache(layers, 64, 16)
    buf = np.zeros(1 << 16, np.uint8)
    base = (buf.ctypes.data + 255) // 256 * 256          # a 256-byte aligned host address
    lib = fa.lib()

    def call(ids, B=2, maxlen=64, ws_bytes=1 << 20, q_off=0, ws_off=0, maxp=16):
        n = len(ids)
        ids_a = (ctypes.c_int32 * max(n, 1))(*ids)
        ptr = (ctypes.c_void_p * max(n, 1))(*([base + q_off] * n))
        lens = base + 4096
        return lib.fa_paged_decode_attn_layers(c._h, n, ids_a, ptr, ptr, maxp, lens, B, maxlen, ptr, None,
                                               base + 8192 + ws_off, ws_bytes, None)

    assert call([]) == fa.ERR_INVALID_ARG                          # n < 1
    assert call([0] * 17) == fa.ERR_INVALID_ARG                    # n > FA_MAX_LAYERS_PER_LAUNCH
    assert call([0, 0]) == fa.ERR_INVALID_ARG                      # a layer twice
    assert call([0, 2]) == fa.ERR_UNSUPPORTED                      # head_dims 256 and 512
    assert call([0, 5]) == fa.ERR_INVALID_ARG                      # layer out of range
    assert call([0, 1], q_off=8) == fa.ERR_INVALID_ARG             # q, out not 16-byte aligned
    assert call([0, 1], maxlen=1000) == fa.ERR_INVALID_ARG         # 16 pages cannot hold 1000 rows
    need = c.decode_layers_workspace_bytes([0, 1], 64, 4096)      # split units need partial rows
    assert need > 0
    assert call([0, 1], B=64, maxlen=4096, maxp=256, ws_bytes=need - 1) == fa.ERR_WORKSPACE   # too small
    assert call([0, 1], B=64, maxlen=4096, maxp=256, ws_bytes=need, ws_off=16) == fa.ERR_INVALID_ARG   # unaligned
    assert call([0, 1], B=0) == fa.OK                              # an empty batch is a no-op


def test_extend_argument_checks(fa):
    """fa_paged_extend_attn / fa_paged_decode_multi_attn refuse what they cannot
    serve before touching the device: negative sizes, query heads per KV head
    that do not divide the 128-row tile, an unbound slab; an empty call is a
    no-op."""
    lib = fa.lib()
    c = fa.Cache([lay(FULL, 256, 6, 2)], 64, 16)     # 3 query heads per KV head: 3 does not divide 128
    assert lib.fa_paged_extend_attn(c._h, 0, None, None, None, None, None, None, 4, 1, 8, 8, 16, None, None,
                                    None) == fa.ERR_UNSUPPORTED
    assert lib.fa_paged_decode_multi_attn(c._h, 0, None, None, None, None, 4, 1, 8, 8, 16, None, None,
                                          None) == fa.ERR_UNSUPPORTED
    c = fa.Cache([lay(SLIDING, 256, 8, 1, 64)], 64, 16)
    assert lib.fa_paged_extend_attn(c._h, 0, None, None, None, None, None, None, 4, -1, 8, 8, 16, None, None,
                                    None) == fa.ERR_INVALID_ARG                       # B < 0
    assert lib.fa_paged_extend_attn(c._h, 0, None, None, None, None, None, None, 4, 0, 0, 0, 0, None, None,
                                    None) == fa.OK                                    # nothing to do
    assert lib.fa_paged_extend_attn(c._h, 0, None, None, None, None, None, None, 4, 1, 8, 8, 16, None, None,
                                    None) == fa.ERR_NOT_BOUND
    assert lib.fa_paged_extend_attn(c._h, 3, None, None, None, None, None, None, 4, 1, 8, 8, 16, None, None,
                                    None) == fa.ERR_INVALID_ARG                       # no layer 3


def test_live_caches_hold_error_word_slots(fa):
    """Each live cache holds one slot of the fixed device array of error
    words: creation beyond FA_MAX_CACHES live descriptors is refused, and a
    destroyed descriptor's slot serves the next one (host only, no GPU)."""
    lib = fa.lib()
    arr = (fa.LayerDesc * 1)(fa._desc(lay(FULL, 512, 8, 1)))
    handles = []
    try:
        while len(handles) <= fa.MAX_CACHES:
            h = ctypes.c_void_p()
            st = lib.fa_cache_create(arr, 1, 8, 16, fa.KV_BF16, ctypes.byref(h))
            if st != fa.OK:
                assert st == fa.ERR_UNSUPPORTED and b"live" in lib.fa_last_error()
                break
            handles.append(h)
        # other tests of this process may hold a few caches
        assert fa.MAX_CACHES - 64 <= len(handles) < fa.MAX_CACHES + 1
        lib.fa_cache_destroy(handles.pop())
        h = ctypes.c_void_p()
        assert lib.fa_cache_create(arr, 1, 8, 16, fa.KV_BF16, ctypes.byref(h)) == fa.OK
        handles.append(h)
    finally:
        for h in handles:
            lib.fa_cache_destroy(h)
    code = ctypes.c_int32()
    assert lib.fa_get_device_error(None, ctypes.byref(code), None) == fa.ERR_INVALID_ARG
