"""Python binding of the GB300 paged-KV attention library.

Argument marshalling only: every step of the store, decode and extend paths
runs in the CUDA kernels of ``libfa_gb300.so`` behind the C ABI declared in
``include/fa.h``.  PyTorch supplies device memory and streams.  Importing this
package raises if the library has not been built; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import weakref

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfa_gb300.so")

FULL, SLIDING = 0, 1
KV_BF16, KV_INT8, KV_FP8 = 0, 1, 2
KV_OWN, KV_AUTO = -1, -2
DEV_ERR_PAGE, DEV_ERR_SLOT, DEV_ERR_BOUND, DEV_ERR_TIMEOUT, DEV_ERR_WORKSPACE, DEV_ERR_RANGE = 1, 2, 4, 8, 16, 32
MAX_CACHES = 4096

FLAG_EARLY_METADATA = 1
FLAG_EXTEND_SPLIT_ALL = 2

NOALLOC_SCRATCH_BYTES = 8 << 20
MAX_LAYERS_PER_LAUNCH = 16

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_NOT_BOUND, ERR_WORKSPACE, ERR_CUDA = 0, 1, 2, 3, 4, 5


class LayerDesc(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("window", ctypes.c_int32), ("kv_source", ctypes.c_int32),
                ("sm_scale", ctypes.c_float)]


class FAError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{_lib.fa_status_string(status).decode()}: {msg}")
        self.status = status


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with full_attention_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    sig = {
        "fa_cache_create": (i32, [ctypes.POINTER(LayerDesc), i32, i32, i32, i32, ctypes.POINTER(vp)]),
        "fa_cache_destroy": (None, [vp]),
        "fa_cache_set_flags": (i32, [vp, ctypes.c_uint32]),
        "fa_cache_set_window_pool": (i32, [vp, i32]),
        "fa_cache_layer_source": (i32, [vp, i32, ctypes.POINTER(i32)]),
        "fa_cache_slab_bytes": (i32, [vp, i32, ctypes.POINTER(sz), ctypes.POINTER(sz)]),
        "fa_cache_bind_slab": (i32, [vp, i32, vp, vp, vp, vp]),
        "fa_kv_bytes_per_token": (sz, [vp, i32]),
        "fa_kv_store": (i32, [vp, i32, vp, vp, vp, i32, vp]),
        "fa_decode_workspace_bytes": (sz, [vp, i32, i32, i32]),
        "fa_extend_workspace_bytes": (sz, []),
        "fa_cache_bind_extend_workspace": (i32, [vp, vp, sz]),
        "fa_paged_decode_attn": (i32, [vp, i32, vp, vp, i32, vp, i32, i32, vp, vp, vp, sz, vp]),
        "fa_paged_decode_store_attn": (i32, [vp, i32, vp, vp, vp, vp, vp, i32, vp, i32, i32, vp, vp, vp, sz, vp]),
        "fa_paged_decode_attn_noalloc": (i32, [vp, i32, vp, vp, i32, vp, i32, i32, vp, vp, vp]),
        "fa_kv_store_layers": (i32, [vp, i32, vp, vp, vp, vp, i32, vp]),
        "fa_paged_decode_multi_attn": (i32, [vp, i32, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp]),
        "fa_decode_layers_workspace_bytes": (sz, [vp, i32, vp, i32, i32]),
        "fa_paged_decode_attn_layers": (i32, [vp, i32, vp, vp, vp, i32, vp, i32, i32, vp, vp, vp, sz, vp]),
        "fa_paged_extend_attn": (i32, [vp, i32, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp]),
        "fa_get_device_error": (i32, [vp, ctypes.POINTER(i32), vp]),
        "fa_last_error": (ctypes.c_char_p, []),
        "fa_status_string": (ctypes.c_char_p, [i32]),
        "fa_version": (i32, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()
_live = weakref.WeakSet()   # every Cache not yet destroyed (for device_error())


def lib() -> ctypes.CDLL:
    return _lib


def _check(status: int) -> None:
    if status != OK:
        raise FAError(status, _lib.fa_last_error().decode())


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _s(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptrs(ts):
    """A host array of device pointers (NULL for None), kept alive by the caller."""
    return (ctypes.c_void_p * len(ts))(*[None if t is None else t.data_ptr() for t in ts])


def _i32s(xs):
    return (ctypes.c_int32 * len(xs))(*[int(x) for x in xs])


def _desc(d: dict) -> LayerDesc:
    return LayerDesc(int(d["kind"]), int(d["head_dim"]), int(d["num_q_heads"]), int(d["num_kv_heads"]),
                     int(d.get("window", 0)), int(d.get("kv_source", KV_OWN)), float(d["sm_scale"]))


class Cache:
    """Host descriptor of a paged KV cache: the layer -> slab map over one page pool.

    `layers` is a list of dicts with the fa_layer_desc fields.  Bound slab
    tensors are referenced here so they outlive the descriptor's use.
    """

    def __init__(self, layers, num_pages: int, page_size: int, kv_dtype: int = KV_BF16):
        self.layers = [dict(d) for d in layers]
        self.num_pages, self.page_size, self.kv_dtype = int(num_pages), int(page_size), int(kv_dtype)
        self.window_pages = 0
        arr = (LayerDesc * len(layers))(*[_desc(d) for d in layers])
        h = ctypes.c_void_p()
        _check(_lib.fa_cache_create(arr, len(layers), self.num_pages, self.page_size, self.kv_dtype,
                                    ctypes.byref(h)))
        self._h = h
        self._slabs = {}
        _live.add(self)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and _lib is not None:
            _lib.fa_cache_destroy(h)
            self._h = None

    def device_error(self, stream=None) -> int:
        """fa_get_device_error: synchronise the stream, then read and clear this
        cache's device error word (FA_DEV_ERR_* bits of its calls' kernels)."""
        code = ctypes.c_int32()
        _check(_lib.fa_get_device_error(self._h, ctypes.byref(code), _s(stream)))
        return code.value

    def set_flags(self, flags: int) -> None:
        """FA_FLAG_* options; FLAG_EARLY_METADATA lets kernels read index
        arrays before the previous kernel in the stream has finished."""
        _check(_lib.fa_cache_set_flags(self._h, int(flags)))

    def set_window_pool(self, window_pages: int) -> None:
        """fa_cache_set_window_pool: the sliding layers' slabs get a pool of
        their own (before binding them)."""
        _check(_lib.fa_cache_set_window_pool(self._h, int(window_pages)))
        self.window_pages = int(window_pages)

    def layer_pages(self, layer: int) -> int:
        """Pages in the slab the layer reads."""
        if self.layers[layer]["kind"] == SLIDING and self.window_pages > 0:
            return self.window_pages
        return self.num_pages

    def source(self, layer: int) -> int:
        out = ctypes.c_int32()
        _check(_lib.fa_cache_layer_source(self._h, layer, ctypes.byref(out)))
        return out.value

    def slab_bytes(self, layer: int):
        kv, sc = ctypes.c_size_t(), ctypes.c_size_t()
        _check(_lib.fa_cache_slab_bytes(self._h, layer, ctypes.byref(kv), ctypes.byref(sc)))
        return kv.value, sc.value

    def bytes_per_token(self, kind: int) -> int:
        return int(_lib.fa_kv_bytes_per_token(self._h, kind))

    def bind(self, layer: int, k, v, k_scale=None, v_scale=None) -> None:
        _check(_lib.fa_cache_bind_slab(self._h, layer, _p(k), _p(v), _p(k_scale), _p(v_scale)))
        self._slabs[layer] = (k, v, k_scale, v_scale)

    def allocate(self, device="cuda") -> dict:
        """Allocate (torch) and bind a slab for every owning layer; returns
        {layer: (k, v, k_scale, v_scale)} with k, v shaped [num_pages][Hkv][page_size][D]."""
        out = {}
        for i, d in enumerate(self.layers):
            if self.source(i) != i:
                continue
            shape = (self.layer_pages(i), d["num_kv_heads"], self.page_size, d["head_dim"])
            # fp8 e4m3 codes are held as raw bytes (uint8 bit patterns)
            dt = {KV_BF16: torch.bfloat16, KV_INT8: torch.int8, KV_FP8: torch.uint8}[self.kv_dtype]
            k = torch.empty(shape, dtype=dt, device=device)
            v = torch.empty(shape, dtype=dt, device=device)
            ks = vs = None
            if self.kv_dtype != KV_BF16:
                ks = torch.empty(shape[:3], dtype=torch.float32, device=device)
                vs = torch.empty(shape[:3], dtype=torch.float32, device=device)
            self.bind(i, k, v, ks, vs)
            out[i] = (k, v, ks, vs)
        return out

    def slab(self, layer: int):
        """(k, v, k_scale, v_scale) tensors the layer reads (its source's for a shared layer)."""
        return self._slabs[self.source(layer)]

    def store(self, layer: int, k, v, slot_mapping, stream=None) -> None:
        _check(_lib.fa_kv_store(self._h, layer, _p(k), _p(v), _p(slot_mapping), int(slot_mapping.numel()),
                                _s(stream)))

    def store_layers(self, layers, ks, vs, slot_mappings, stream=None) -> None:
        """fa_kv_store_layers: the stores of several layers in one launch
        (shared layers are skipped)."""
        T = int(slot_mappings[0].numel())
        _check(_lib.fa_kv_store_layers(self._h, len(layers), _i32s(layers), _ptrs(ks), _ptrs(vs),
                                       _ptrs(slot_mappings), T, _s(stream)))

    def decode_layers_workspace_bytes(self, layers, batch: int, max_seq_len: int) -> int:
        return int(_lib.fa_decode_layers_workspace_bytes(self._h, len(layers), _i32s(layers), batch, max_seq_len))

    def decode_layers(self, layers, qs, block_tables, seq_lens, max_seq_len: int, outs, lses=None,
                      workspace=None, stream=None) -> None:
        """fa_paged_decode_attn_layers: decode several layers of one head_dim
        in one launch (the current rows must already be stored)."""
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        _check(_lib.fa_paged_decode_attn_layers(self._h, len(layers), _i32s(layers), _ptrs(qs), _ptrs(block_tables),
                                                int(block_tables[0].shape[1]), _p(seq_lens), int(qs[0].shape[0]),
                                                int(max_seq_len), _ptrs(outs), None if lses is None else _ptrs(lses),
                                                _p(workspace), ws_bytes, _s(stream)))

    def decode_workspace_bytes(self, layer: int, batch: int, max_seq_len: int) -> int:
        return int(_lib.fa_decode_workspace_bytes(self._h, layer, batch, max_seq_len))

    def bind_extend_workspace(self, workspace) -> None:
        """fa_cache_bind_extend_workspace: let extend and multi-token decode
        calls split their last wave through `workspace` (a device tensor of at
        least extend_workspace_bytes() bytes; None unbinds).  The tensor is
        kept referenced while bound."""
        nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        _check(_lib.fa_cache_bind_extend_workspace(self._h, _p(workspace), nbytes))
        self._extend_ws = workspace

    def decode(self, layer: int, q, block_table, seq_lens, max_seq_len: int, out, lse=None, workspace=None,
               stream=None) -> None:
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        _check(_lib.fa_paged_decode_attn(self._h, layer, _p(q), _p(block_table), int(block_table.shape[1]),
                                         _p(seq_lens), int(q.shape[0]), int(max_seq_len), _p(out), _p(lse),
                                         _p(workspace), ws_bytes, _s(stream)))

    def decode_store(self, layer: int, q, k_new, v_new, slot_mapping, block_table, seq_lens, max_seq_len: int,
                     out, lse=None, workspace=None, stream=None) -> None:
        """fa_paged_decode_store_attn: store the current token's k, v rows and
        decode in one launch (owning layers; a shared layer only decodes)."""
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        _check(_lib.fa_paged_decode_store_attn(self._h, layer, _p(q), _p(k_new), _p(v_new), _p(slot_mapping),
                                               _p(block_table), int(block_table.shape[1]), _p(seq_lens),
                                               int(q.shape[0]), int(max_seq_len), _p(out), _p(lse), _p(workspace),
                                               ws_bytes, _s(stream)))

    def decode_noalloc(self, layer: int, q, block_table, seq_lens, max_seq_len: int, out, lse=None,
                       stream=None) -> None:
        """fa_paged_decode_attn_noalloc: decode with the library's fixed scratch
        (no device allocation); calls must not overlap on the GPU."""
        _check(_lib.fa_paged_decode_attn_noalloc(self._h, layer, _p(q), _p(block_table), int(block_table.shape[1]),
                                                 _p(seq_lens), int(q.shape[0]), int(max_seq_len), _p(out), _p(lse),
                                                 _s(stream)))

    def decode_multi(self, layer: int, q, qo_indptr, seq_lens, block_table, max_q_len: int, max_seq_len: int, out,
                     lse=None, stream=None) -> None:
        """fa_paged_decode_multi_attn: several new tokens per sequence, their rows
        already stored; every key from the slab."""
        _check(_lib.fa_paged_decode_multi_attn(self._h, layer, _p(q), _p(qo_indptr), _p(seq_lens), _p(block_table),
                                               int(block_table.shape[1]), int(seq_lens.numel()), int(q.shape[0]),
                                               int(max_q_len), int(max_seq_len), _p(out), _p(lse), _s(stream)))

    def extend(self, layer: int, q, k_ext, v_ext, qo_indptr, prefix_lens, block_table, max_q_len: int,
               max_prefix_len: int, out, lse=None, stream=None) -> None:
        maxp = int(block_table.shape[1]) if block_table is not None else 0
        _check(_lib.fa_paged_extend_attn(self._h, layer, _p(q), _p(k_ext), _p(v_ext), _p(qo_indptr),
                                         _p(prefix_lens), _p(block_table), maxp, int(prefix_lens.numel()),
                                         int(q.shape[0]), int(max_q_len), int(max_prefix_len), _p(out), _p(lse),
                                         _s(stream)))


def device_error(stream=None) -> int:
    """The OR of every live cache's device error word, each read and cleared
    (Cache.device_error) after synchronising the stream."""
    code = 0
    for c in list(_live):
        if getattr(c, "_h", None) is not None:
            code |= c.device_error(stream)
    return code


def workspace(nbytes: int, device="cuda"):
    """A zeroed, 256-byte-aligned decode workspace of at least nbytes
    (torch-allocated; decode calls leave its counters zero for reuse)."""
    return torch.zeros(max(int(nbytes), 1), dtype=torch.uint8, device=device)


def extend_workspace_bytes() -> int:
    """fa_extend_workspace_bytes: the extend split workspace's size on the
    current device."""
    return int(_lib.fa_extend_workspace_bytes())
