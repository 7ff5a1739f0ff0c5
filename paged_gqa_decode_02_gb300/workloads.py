"""Seeded synthetic inputs for paged GQA decode.

This module only draws random numbers and lays out block tables. It holds
none of the method's arithmetic (no quantisation, no attention, no
logical-to-physical addressing of token slots); both the CUDA path and the
CPU oracle consume what it returns.

Workload shapes follow the pages' decode workloads:
  * the Qwen2.5-7B layer of "从零实现 C++ LLM 推理引擎" (28 Q heads sharing
    4 KV heads, head_dim 128; section "3. GQA"),
  * a Qwen3-8B-shaped int8-KV case, a long-context uint4 case and a
    continuous-batching mix with prefix sharing, which exercise the paged
    cache, int8/uint4 KV quantisation and prefix cache of the heterogeneous
    engine article (sections 2.3-2.5, 4.3, 4.7).

No public dataset or model is involved: N(0, 1) activations stand in for
real ones.

Random streams: ``numpy.random.default_rng([seed, stream])`` with stream
0 = sequence lengths, 1 = q, 2 = K, 3 = V, 4 = per-channel offsets,
5 = physical block permutation, 6 = the queries of several tokens per
sequence. Values are drawn in float32 and rounded to
bfloat16 with round-to-nearest-even.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np

KV_DTYPES = ("bf16", "uint8", "uint4")
# every storage format a case may name; random cases draw from KV_DTYPES
ALL_KV_DTYPES = KV_DTYPES + ("fp8",)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns (uint16), round-to-nearest-even.

    Inputs are finite by construction (normal draws)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    # finite inputs stay below 0xFF800000 + 0x8000: no uint32 overflow
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns -> float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass
class AppendCall:
    """One call of the append entry point: new tokens for each sequence."""

    k_bits: np.ndarray  # uint16 [T_new, Hkv, D]
    v_bits: np.ndarray  # uint16 [T_new, Hkv, D]
    cu_new: np.ndarray  # int32 [B'+1]: new tokens of sequence i are rows cu[i]..cu[i+1]
    ctx_lens: np.ndarray  # int32 [B']: tokens already stored before this call
    block_table: np.ndarray  # int32 [B', max_blocks]

    @property
    def batch(self) -> int:
        return int(self.ctx_lens.shape[0])

    @property
    def max_new(self) -> int:
        if self.batch == 0:
            return 0
        return int(np.max(np.diff(self.cu_new)))


@dataclasses.dataclass
class Workload:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    kv_dtype: str
    num_blocks: int
    seq_lens: np.ndarray  # int32 [B]
    block_table: np.ndarray  # int32 [B, max_blocks]; unused entries are -1
    q_bits: np.ndarray  # uint16 [B, Hq, D]
    k_bits: np.ndarray  # uint16 [sum(seq_lens), Hkv, D], sequence-major
    v_bits: np.ndarray  # uint16 [sum(seq_lens), Hkv, D]
    tok_off: np.ndarray  # int64 [B+1]: tokens of sequence b are rows tok_off[b]..tok_off[b+1]
    softmax_scale: float
    # prefix sharing: number of leading logical blocks of sequence b that map
    # to blocks shared with its group (0 = none), and the shared groups
    shared_blocks: np.ndarray = None  # int32 [B]
    groups: list = None  # list of (member indices, shared physical ids, prefix k bits, prefix v bits)

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def group_size(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def n_blocks_of(self, b: int) -> int:
        return -(-int(self.seq_lens[b]) // self.block_size)

    def fill_calls(self, leave_last: bool = True) -> List[AppendCall]:
        """Append calls that load every sequence's cached tokens into an empty pool.

        With ``leave_last`` each sequence's final token is left out, so that
        ``step_call()`` appends it (one decode step: store, then attend).
        Shared prefix blocks are written once, by one extra sequence per group
        whose table row holds just the group's shared blocks; members append
        only their private tokens (their context already covers the prefix).
        """
        B, MB = self.batch, self.max_blocks
        rows_k, rows_v, cu, ctx, tabs = [], [], [0], [], []
        if self.groups:
            for members, shared_ids, pk, pv in self.groups:
                row = np.full(MB, -1, np.int32)
                row[: len(shared_ids)] = shared_ids
                rows_k.append(pk)
                rows_v.append(pv)
                cu.append(cu[-1] + pk.shape[0])
                ctx.append(0)
                tabs.append(row)
        for b in range(B):
            s = int(self.seq_lens[b])
            end = s - 1 if (leave_last and s > 0) else s
            start = int(self.shared_blocks[b]) * self.block_size if self.shared_blocks is not None else 0
            start = min(start, end)
            o = int(self.tok_off[b])
            rows_k.append(self.k_bits[o + start: o + end])
            rows_v.append(self.v_bits[o + start: o + end])
            cu.append(cu[-1] + (end - start))
            ctx.append(start)
            tabs.append(self.block_table[b])
        Hkv, D = self.num_kv_heads, self.head_dim
        k = np.concatenate(rows_k) if rows_k else np.zeros((0, Hkv, D), np.uint16)
        v = np.concatenate(rows_v) if rows_v else np.zeros((0, Hkv, D), np.uint16)
        return [AppendCall(np.ascontiguousarray(k), np.ascontiguousarray(v),
                           np.asarray(cu, np.int32), np.asarray(ctx, np.int32),
                           np.ascontiguousarray(np.stack(tabs).astype(np.int32)))]

    def step_call(self, n_new: int = 1) -> AppendCall:
        """The decode step's append: the last token of every non-empty
        sequence (with n_new > 1: its last n_new tokens, or all it has)."""
        B = self.batch
        cnt = np.minimum(self.seq_lens.astype(np.int64), n_new)
        sel = [int(self.tok_off[b]) + int(self.seq_lens[b]) - int(cnt[b]) + i for b in range(B) for i in range(int(cnt[b]))]
        k = self.k_bits[sel] if sel else np.zeros((0, self.num_kv_heads, self.head_dim), np.uint16)
        v = self.v_bits[sel] if sel else np.zeros((0, self.num_kv_heads, self.head_dim), np.uint16)
        cu = np.concatenate([[0], np.cumsum(cnt)]).astype(np.int32)
        ctx = (self.seq_lens - cnt).astype(np.int32)
        return AppendCall(np.ascontiguousarray(k), np.ascontiguousarray(v), cu, ctx,
                          np.ascontiguousarray(self.block_table))

    def unique_blocks(self) -> int:
        """Distinct physical blocks referenced by the decode tables."""
        t = self.block_table
        return int(np.unique(t[t >= 0]).size)


def _draw_tokens(rng, n, Hkv, D, offset=None):
    x = rng.standard_normal((n, Hkv, D), dtype=np.float32)
    if offset is not None:
        x += offset[None, :, :]
    return f32_to_bf16_bits(x)


def _assign_blocks(n_blocks_per_seq, num_blocks, rng_perm, max_blocks):
    """Map every (sequence, logical block) to a distinct physical block, in
    (sequence, logical) order, taking ids from a seeded permutation."""
    perm = rng_perm.permutation(num_blocks).astype(np.int32)
    B = len(n_blocks_per_seq)
    table = np.full((B, max_blocks), -1, np.int32)
    pos = 0
    for b, nb in enumerate(n_blocks_per_seq):
        table[b, :nb] = perm[pos: pos + nb]
        pos += nb
    return table


def make_case(name, seed, batch, num_q_heads, num_kv_heads, head_dim, block_size, kv_dtype,
              seq_lens, extra_blocks=0, channel_offset_sigma=None, max_blocks=None,
              softmax_scale=None) -> Workload:
    """Generic seeded case with private (unshared) blocks."""
    assert kv_dtype in ALL_KV_DTYPES
    seq_lens = np.asarray(seq_lens, np.int32)
    assert seq_lens.shape == (batch,)
    nbs = [-(-int(s) // block_size) for s in seq_lens]
    num_blocks = max(1, sum(nbs) + int(extra_blocks))
    if max_blocks is None:
        max_blocks = max(1, max(nbs) if nbs else 1)
    rng_q = np.random.default_rng([seed, 1])
    rng_k = np.random.default_rng([seed, 2])
    rng_v = np.random.default_rng([seed, 3])
    rng_off = np.random.default_rng([seed, 4])
    rng_perm = np.random.default_rng([seed, 5])
    off_k = off_v = None
    if channel_offset_sigma is not None:
        off_k = (rng_off.standard_normal((num_kv_heads, head_dim), dtype=np.float32)
                 * np.float32(channel_offset_sigma))
        off_v = (rng_off.standard_normal((num_kv_heads, head_dim), dtype=np.float32)
                 * np.float32(channel_offset_sigma))
    table = _assign_blocks(nbs, num_blocks, rng_perm, max_blocks)
    q = f32_to_bf16_bits(rng_q.standard_normal((batch, num_q_heads, head_dim), dtype=np.float32))
    ks = [_draw_tokens(rng_k, int(s), num_kv_heads, head_dim, off_k) for s in seq_lens]
    vs = [_draw_tokens(rng_v, int(s), num_kv_heads, head_dim, off_v) for s in seq_lens]
    k = np.concatenate(ks) if ks else np.zeros((0, num_kv_heads, head_dim), np.uint16)
    v = np.concatenate(vs) if vs else np.zeros((0, num_kv_heads, head_dim), np.uint16)
    tok_off = np.concatenate([[0], np.cumsum(seq_lens.astype(np.int64))])
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(head_dim)
    return Workload(name, batch, num_q_heads, num_kv_heads, head_dim, block_size, kv_dtype,
                    num_blocks, seq_lens, table, q, k, v, tok_off,
                    float(np.float32(softmax_scale)),
                    shared_blocks=np.zeros(batch, np.int32), groups=None)


def multi_token_queries(seed: int, batch: int, n_q: int, num_q_heads: int, head_dim: int) -> np.ndarray:
    """Query rows of several new tokens per sequence (chunked prefill or
    speculative verification), bf16 bits [batch, n_q, Hq, D] from stream 6."""
    rng = np.random.default_rng([seed, 6])
    return f32_to_bf16_bits(rng.standard_normal((batch, n_q, num_q_heads, head_dim), dtype=np.float32))


def tiny(seed: int = 1) -> Workload:
    """batch 2, 4 Q / 2 KV heads, head_dim 64, block 16, seq_lens {37, 5},
    a pool of 8 physical blocks (the 4 used ones taken from a seeded
    permutation; the other 4 stay unused), bf16 KV, scale 1/8."""
    return make_case("tiny", seed, 2, 4, 2, 64, 16, "bf16", [37, 5], extra_blocks=4)


def qwen25_7b(seed: int = 2) -> Workload:
    """batch 32, 28 Q / 4 KV heads, head_dim 128, block 16, seq_lens uniform
    in [512, 4096], pool sized to exactly the blocks in use, bf16 KV."""
    rng = np.random.default_rng([seed, 0])
    seq = rng.integers(512, 4097, size=32).astype(np.int32)
    return make_case("qwen25_7b_bf16", seed, 32, 28, 4, 128, 16, "bf16", seq)


def qwen3_8b_int8(seed: int = 3) -> Workload:
    """batch 64, 32 Q / 8 KV heads, head_dim 128, block 16, seq_lens uniform
    in [1, 8192]; K and V are N(0,1) plus a per-(kv head, channel) offset
    drawn from N(0, 0.5), stored as uint8 codes."""
    rng = np.random.default_rng([seed, 0])
    seq = rng.integers(1, 8193, size=64).astype(np.int32)
    return make_case("qwen3_8b_int8", seed, 64, 32, 8, 128, 16, "uint8", seq,
                     channel_offset_sigma=0.5)


def qwen3_8b_fp8(seed: int = 3) -> Workload:
    """The Qwen3-8B-shaped case (same lengths and values as the uint8 one)
    stored as fp8 (E4M3) codes."""
    rng = np.random.default_rng([seed, 0])
    seq = rng.integers(1, 8193, size=64).astype(np.int32)
    return make_case("qwen3_8b_fp8", seed, 64, 32, 8, 128, 16, "fp8", seq,
                     channel_offset_sigma=0.5)


def long_uint4(seed: int = 4) -> Workload:
    """batch 4, 32 Q / 8 KV heads, head_dim 128, block 32, 32768 tokens per
    sequence, stored as packed uint4 codes."""
    return make_case("long_uint4", seed, 4, 32, 8, 128, 32, "uint4", [32768] * 4)


def prefix_mix(seed: int = 5, batch: int = 256, n_groups: int = 8, prefix_tokens: int = 512,
               median: float = 1000.0, sigma: float = 1.0, max_len: int = 32768) -> Workload:
    """Continuous-batching mix with a prefix cache: batch 256, 28 Q / 4 KV
    heads, head_dim 128, block 16, seq_lens lognormal (median 1000, sigma 1)
    clipped to [1, 32768]; 8 groups of 32 consecutive sequences share the
    physical blocks of their first 512 tokens.

    A member shares only full blocks that lie before the block holding its
    last token (a partially filled tail block is private, as after
    copy-on-write), so every decode-step append writes a private block."""
    Hq, Hkv, D, bs = 28, 4, 128, 16
    rng = np.random.default_rng([seed, 0])
    seq = np.clip(np.rint(rng.lognormal(math.log(median), sigma, size=batch)), 1, max_len).astype(np.int32)
    per_group = batch // n_groups
    n_prefix_blocks = prefix_tokens // bs
    nbs = [-(-int(s) // bs) for s in seq]
    shared = np.array([min(n_prefix_blocks, (int(s) - 1) // bs) for s in seq], np.int32)
    private = [nb - sh for nb, sh in zip(nbs, shared)]
    num_blocks = n_groups * n_prefix_blocks + sum(private)
    max_blocks = max(nbs)
    rng_q = np.random.default_rng([seed, 1])
    rng_k = np.random.default_rng([seed, 2])
    rng_v = np.random.default_rng([seed, 3])
    rng_perm = np.random.default_rng([seed, 5])
    perm = rng_perm.permutation(num_blocks).astype(np.int32)
    table = np.full((batch, max_blocks), -1, np.int32)
    pos = 0
    groups = []
    for gi in range(n_groups):
        ids = perm[pos: pos + n_prefix_blocks]
        pos += n_prefix_blocks
        pk = _draw_tokens(rng_k, prefix_tokens, Hkv, D)
        pv = _draw_tokens(rng_v, prefix_tokens, Hkv, D)
        members = list(range(gi * per_group, (gi + 1) * per_group))
        groups.append((members, ids, pk, pv))
    for b in range(batch):
        nsh = int(shared[b])
        g = groups[b // per_group]
        table[b, :nsh] = g[1][:nsh]
        table[b, nsh: nbs[b]] = perm[pos: pos + private[b]]
        pos += private[b]
    assert pos == num_blocks
    q = f32_to_bf16_bits(rng_q.standard_normal((batch, Hq, D), dtype=np.float32))
    ks, vs = [], []
    for b in range(batch):
        g = groups[b // per_group]
        n_sh_tok = int(shared[b]) * bs
        own = int(seq[b]) - n_sh_tok
        ks.append(np.concatenate([g[2][:n_sh_tok], _draw_tokens(rng_k, own, Hkv, D)]))
        vs.append(np.concatenate([g[3][:n_sh_tok], _draw_tokens(rng_v, own, Hkv, D)]))
    tok_off = np.concatenate([[0], np.cumsum(seq.astype(np.int64))])
    return Workload("prefix_mix", batch, Hq, Hkv, D, bs, "bf16", num_blocks, seq, table, q,
                    np.concatenate(ks), np.concatenate(vs), tok_off,
                    float(np.float32(1.0 / math.sqrt(D))), shared_blocks=shared, groups=groups)


CONFIGS = {
    "tiny": tiny,
    "qwen25_7b_bf16": qwen25_7b,
    "qwen3_8b_int8": qwen3_8b_int8,
    "long_uint4": long_uint4,
    "qwen3_8b_fp8": qwen3_8b_fp8,
    "prefix_mix": prefix_mix,
}


def random_small(seed: int, kv_dtype: Optional[str] = None) -> Workload:
    """A small random case (B <= 3, head_dim in {64, 128}, block in {16, 32},
    seq_len <= 70, GQA group in {1, 2, 4, 7}) for quick parity sweeps."""
    rng = np.random.default_rng([1000 + seed, 0])
    B = int(rng.integers(1, 4))
    D = int(rng.choice([64, 128]))
    bs = int(rng.choice([16, 32]))
    Hkv = int(rng.choice([1, 2]))
    g = int(rng.choice([1, 2, 4, 7]))
    dt = kv_dtype or str(rng.choice(KV_DTYPES))
    seq = rng.integers(1, 71, size=B).astype(np.int32)
    return make_case(f"random{seed}", 1000 + seed, B, Hkv * g, Hkv, D, bs, dt, seq,
                     extra_blocks=int(rng.integers(0, 4)),
                     channel_offset_sigma=0.5 if dt != "bf16" else None)
