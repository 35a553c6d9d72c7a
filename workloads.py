"""Seeded synthetic workloads for Gemma-4-style paged-KV attention.

This module only describes and generates inputs: layer layouts, sequence
lengths, page pools, block tables, slot mappings and N(0,1) bf16 tensors.
It holds none of the attention, store or quantisation arithmetic, so both the
CUDA path and the fp64 oracle can take their inputs from it without sharing
any computation.

The five workloads mirror the decode/extend regimes the pages describe:
full-attention layers (causal, head_dim 512) and sliding layers (causal and
q_pos - kv_pos < W, head_dim 256), with KV-shared layers that read an earlier
owning layer's slab ("FreeToken PR #898: read the source layer's kv slab on
kv-shared layers", description).  Layer layout for the 12-layer decode
workloads: kinds S S S S F S S S S F S S (a full layer every fifth layer, as in
the E2B-style models), layers 0-6 own a slab and 7-11 are KV-shared; each
shared layer's source is resolved by the library/oracle from the rule (the
last earlier owning layer of the same kind).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

FULL = 0
SLIDING = 1
KV_OWN = -1   # the layer owns a slab
KV_AUTO = -2  # shared layer: source = last earlier owning layer of its kind

KV_BF16 = 0
KV_INT8 = 1
KV_FP8 = 2


def layer(kind: int, head_dim: int, hq: int, hkv: int, window: int = 0,
          kv_source: int = KV_OWN) -> dict:
    """One layer descriptor (plain dict; the binding and the oracle both read it)."""
    return dict(kind=kind, head_dim=head_dim, num_q_heads=hq, num_kv_heads=hkv,
                window=window if kind == SLIDING else 0, kv_source=kv_source,
                sm_scale=float(np.float32(1.0 / math.sqrt(head_dim))))


def layout_12(hq: int, hkv: int, window: int) -> list[dict]:
    """12 layers, kinds S S S S F S S S S F S S; 0-6 own, 7-11 shared."""
    kinds = "SSSSFSSSSFSS"
    out = []
    for i, c in enumerate(kinds):
        src = KV_OWN if i < 7 else KV_AUTO
        if c == "F":
            out.append(layer(FULL, 512, hq, hkv, 0, src))
        else:
            out.append(layer(SLIDING, 256, hq, hkv, window, src))
    return out


@dataclass
class DecodeWorkload:
    name: str
    seed: int
    batch: int
    ctx_lo: int
    ctx_hi: int
    page_size: int
    layers: list
    kv_dtype: int = KV_BF16
    pool_factor: float = 1.25
    min_pool_pages: int = 0
    # sliding layers get their own table holding only in-window pages (-1 below)
    sliding_window_table: bool = False
    fixed_lens: list | None = None


@dataclass
class ExtendWorkload:
    name: str
    seed: int
    batch: int
    prompt_len: int
    chunk: int
    page_size: int
    layers: list
    kv_dtype: int = KV_BF16
    pool_factor: float = 1.25


def tiny_decode() -> DecodeWorkload:
    """1 sequence, context 200, page 16, 32 permuted pages, 4 q / 1 KV head;
    a sliding layer (D 256, W 64), a full layer (D 512) and a shared layer
    reading the sliding layer's slab."""
    layers = [layer(SLIDING, 256, 4, 1, 64), layer(FULL, 512, 4, 1),
              layer(SLIDING, 256, 4, 1, 64, KV_AUTO)]
    return DecodeWorkload("tiny decode (B=1, ctx 200, 4q/1kv, S D256 W64 + F D512 + shared)",
                          0, 1, 200, 200, 16, layers, min_pool_pages=32, fixed_lens=[200])


def e2b_decode() -> DecodeWorkload:
    return DecodeWorkload("E2B-like decode (B=64, ctx U[512,4096], 8q/1kv, S D256 W512 / F D512, "
                          "7 owning + 5 shared layers, bf16)",
                          1, 64, 512, 4096, 16, layout_12(8, 1, 512))


def chunked_prefill() -> ExtendWorkload:
    layers = [layer(SLIDING, 256, 16, 8, 1024), layer(FULL, 512, 16, 2)]
    return ExtendWorkload("chunked prefill (4 x 4096-token prompts in 512-token chunks; "
                          "S 16q/8kv D256 W1024, F 16q/2kv D512)", 2, 4, 4096, 512, 16, layers)


def long_decode() -> DecodeWorkload:
    return DecodeWorkload("long-context decode (B=8, ctx U[32768,131072], 8q/1kv, S D256 W1024 "
                          "in-window pages only / F D512)", 3, 8, 32768, 131072, 16,
                          layout_12(8, 1, 1024), sliding_window_table=True)


def int8_decode() -> DecodeWorkload:
    return DecodeWorkload("int8 per-token-head KV decode (B=128, ctx U[1024,8192], 8q/1kv, "
                          "S D256 W1024 / F D512)", 4, 128, 1024, 8192, 16,
                          layout_12(8, 1, 1024), kv_dtype=KV_INT8)


def fp8_decode() -> DecodeWorkload:
    """The int8 decode workload's shapes with the fp8 e4m3 per-token-head format."""
    return DecodeWorkload("fp8 e4m3 per-token-head KV decode (B=128, ctx U[1024,8192], 8q/1kv, "
                          "S D256 W1024 / F D512)", 4, 128, 1024, 8192, 16,
                          layout_12(8, 1, 1024), kv_dtype=KV_FP8)


ALL = {"tiny_decode": tiny_decode, "e2b_decode": e2b_decode,
       "chunked_prefill": chunked_prefill, "long_decode": long_decode,
       "int8_decode": int8_decode, "fp8_decode": fp8_decode}


# ---------------------------------------------------------------------------
# generators
# ---------------------------------------------------------------------------

def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def seq_lens(w: DecodeWorkload) -> np.ndarray:
    if w.fixed_lens is not None:
        return np.asarray(w.fixed_lens, dtype=np.int32)
    return rng(w.seed).integers(w.ctx_lo, w.ctx_hi + 1, size=w.batch).astype(np.int32)


@dataclass
class PagePlan:
    """Physical page assignment for one group of layers sharing a block table."""
    num_pages: int
    block_table: np.ndarray        # int32 [B][max_pages], -1 where no page is assigned
    first_page: np.ndarray = field(default=None)  # int32 [B], first logical page assigned


def plan_pages(lens: np.ndarray, page_size: int, seed: int, pool_factor: float = 1.25,
               min_pool: int = 0, window: int = 0, max_pages: int | None = None) -> PagePlan:
    """Assign logical pages of each sequence to a seeded random permutation of a
    pool about pool_factor x the pages needed.  With window > 0 only the pages
    that hold positions [max(0, L - window), L - 1] get a page; the others stay -1."""
    r = rng(seed * 7919 + 17 + window)
    B = len(lens)
    need_hi = [(int(L) + page_size - 1) // page_size for L in lens]
    need_lo = [0] * B
    if window > 0:
        need_lo = [max(0, int(L) - window) // page_size for L in lens]
    total = sum(h - l for h, l in zip(need_hi, need_lo))
    pool = max(min_pool, int(math.ceil(total * pool_factor)), 1)
    perm = r.permutation(pool).astype(np.int32)
    maxp = max_pages if max_pages is not None else max(max(need_hi), 1)
    bt = np.full((B, maxp), -1, dtype=np.int32)
    k = 0
    for b in range(B):
        for p in range(need_lo[b], need_hi[b]):
            bt[b, p] = perm[k]
            k += 1
    return PagePlan(pool, bt, np.asarray(need_lo, dtype=np.int32))


def decode_slot_mapping(lens: np.ndarray, block_table: np.ndarray, page_size: int) -> np.ndarray:
    """Slot of the current token (position L-1) of each sequence: page * ps + off."""
    out = np.full(len(lens), -1, dtype=np.int32)   # -1: nothing to store (empty sequence)
    for b, L in enumerate(lens):
        if int(L) <= 0:
            continue
        pos = int(L) - 1
        out[b] = block_table[b, pos // page_size] * page_size + pos % page_size
    return out


def slots_for_positions(block_table_row: np.ndarray, positions: np.ndarray, page_size: int) -> np.ndarray:
    pages = block_table_row[positions // page_size].astype(np.int64)
    return (pages * page_size + positions % page_size).astype(np.int32)


def randn_bf16(shape, seed: int, device="cpu"):
    """N(0,1) values rounded to bf16, from a seeded torch generator."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return torch.randn(*shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def bf16_bits(t) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (what the oracle reads)."""
    import torch
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
