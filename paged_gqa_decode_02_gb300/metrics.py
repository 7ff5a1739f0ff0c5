"""Byte accounting for the decode roofline.

Algorithmic bytes of one decode call: K and V of every valid token (codes,
counted per token, not per page), the scale (and zero-point) metadata of
every touched (block, kv head) for quantised pools, q, out, the block-table entries
read and the sequence lengths. A physical block shared by several sequences
(prefix cache) is counted once.
"""
from __future__ import annotations

import numpy as np

ELEM_BITS = {"bf16": 16, "uint8": 8, "uint4": 4, "fp8": 8}
# metadata bytes per channel of a touched (block, kv head), K and V together:
# f32 scale + i32 zero point for the integer formats, f32 scale for fp8
META_BYTES = {"bf16": 0, "uint8": 16, "uint4": 16, "fp8": 8}


def decode_bytes(wl, n_q: int = 1) -> dict:
    """Byte counts of one decode call (n_q query tokens per sequence)."""
    bs, D, Hkv = wl.block_size, wl.head_dim, wl.num_kv_heads
    bits = ELEM_BITS[wl.kv_dtype]
    # valid tokens per physical block (max over the sequences that use it)
    valid = {}
    logical_tokens = 0
    for b in range(wl.batch):
        n = int(wl.seq_lens[b])
        logical_tokens += n
        for lp in range(-(-n // bs)):
            phys = int(wl.block_table[b, lp])
            v = min(bs, n - lp * bs)
            if valid.get(phys, 0) < v:
                valid[phys] = v
    unique_tokens = sum(valid.values())
    per_token = 2 * Hkv * D * bits // 8  # K and V, all kv heads
    meta_per_block = Hkv * D * META_BYTES[wl.kv_dtype]
    pages = sum(-(-int(s) // bs) for s in wl.seq_lens)
    q = wl.batch * n_q * wl.num_q_heads * D * 2
    out = wl.batch * n_q * wl.num_q_heads * D * 4
    tables = pages * 4 + wl.batch * 4
    kv_unique = unique_tokens * per_token + len(valid) * meta_per_block
    kv_logical = logical_tokens * per_token + pages * meta_per_block
    return {
        "algorithmic": kv_unique + q + out + tables,
        "logical": kv_logical + q + out + tables,
        "kv_unique": kv_unique,
        "tokens_scanned": logical_tokens,
        "unique_blocks": len(valid),
        "pages": pages,
    }
