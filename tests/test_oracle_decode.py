"""Pins for the oracle's decode attention (CPU only).

The oracle computes the plain definition (paged_attention_kernel of the
heterogeneous engine article, section 4.3: gather through the page table,
dequantise, score / sqrt(head_dim), softmax, P.V, normalise) with query head h
reading KV head h / (Hq/Hkv) (repeat_kv grouping of the Qwen2.5-7B engine
article, section "3. GQA"). These tests pin it to things other than itself:
an independent dense numpy attention on gathered contiguous K/V, closed
forms, and invariances.
"""
import math

import numpy as np
import pytest

from oracle import oracle
from paged_gqa_decode_02_gb300 import workloads as W


def _load(wl, leave_last=True):
    pool = oracle.OraclePool(wl.kv_dtype, wl.num_blocks, wl.num_kv_heads, wl.block_size,
                             wl.head_dim, fill=0x7FC0 if wl.kv_dtype == "bf16" else 0)
    calls = wl.fill_calls(leave_last=leave_last)
    if leave_last:
        calls.append(wl.step_call())
    for c in calls:
        assert pool.append_call(c) == 0
    return pool


def _dense_reference(q, Ks, Vs, scale, Hkv):
    """softmax(q K^T * scale) V per (b, h) on contiguous per-sequence K/V,
    written with numpy float64 matrix products and repeat_kv expansion."""
    B, Hq, D = q.shape
    g = Hq // Hkv
    out = np.zeros((B, Hq, D))
    for b in range(B):
        K, V = Ks[b], Vs[b]  # [n, Hkv, D]
        if K.shape[0] == 0:
            continue
        Kx = np.repeat(K, g, axis=1).transpose(1, 0, 2)  # [Hq, n, D]
        Vx = np.repeat(V, g, axis=1).transpose(1, 0, 2)
        s = np.einsum("hd,hnd->hn", q[b], Kx) * scale
        s -= s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p /= p.sum(axis=1, keepdims=True)
        out[b] = np.einsum("hn,hnd->hd", p, Vx)
    return out


def _seq_kv(wl, b):
    o, n = int(wl.tok_off[b]), int(wl.seq_lens[b])
    return (W.bf16_bits_to_f32(wl.k_bits[o:o + n]).astype(np.float64),
            W.bf16_bits_to_f32(wl.v_bits[o:o + n]).astype(np.float64))


@pytest.mark.parametrize("seed", range(6))
def test_bf16_decode_matches_dense_attention(seed):
    wl = W.random_small(seed, "bf16")
    pool = _load(wl)
    out, st = pool.decode(wl.q_bits, wl.block_table, wl.seq_lens, wl.softmax_scale)
    assert st == 0
    q = W.bf16_bits_to_f32(wl.q_bits).astype(np.float64)
    kv = [_seq_kv(wl, b) for b in range(wl.batch)]
    ref = _dense_reference(q, [k for k, _ in kv], [v for _, v in kv], wl.softmax_scale,
                           wl.num_kv_heads)
    np.testing.assert_allclose(out.reshape(ref.shape), ref, rtol=1e-12, atol=1e-12)


def test_tiny_config_matches_dense_attention():
    wl = W.tiny()
    assert wl.softmax_scale == 0.125 and wl.num_blocks == 8
    pool = _load(wl)
    out, st = pool.decode(wl.q_bits, wl.block_table, wl.seq_lens, wl.softmax_scale)
    assert st == 0
    q = W.bf16_bits_to_f32(wl.q_bits).astype(np.float64)
    kv = [_seq_kv(wl, b) for b in range(wl.batch)]
    ref = _dense_reference(q, [k for k, _ in kv], [v for _, v in kv], 0.125, 2)
    np.testing.assert_allclose(out.reshape(ref.shape), ref, rtol=1e-12, atol=1e-12)
    # unused blocks hold NaN and must never be read
    assert np.isfinite(out).all()


@pytest.mark.parametrize("dt", ["uint8", "uint4"])
def test_quantised_decode_matches_dense_on_dequantised_codes(dt):
    wl = W.random_small(21, dt)
    pool = _load(wl)
    out, st = pool.decode(wl.q_bits, wl.block_table, wl.seq_lens, wl.softmax_scale)
    assert st == 0
    bs, D = wl.block_size, wl.head_dim

    def deq(codes, sc, zp, b, n):
        t = np.arange(n)
        phys = wl.block_table[b, t // bs]
        if dt == "uint8":
            c = codes[phys, :, t % bs, :].astype(np.float64)
        else:
            by = codes[phys, :, t % bs, :]
            c = np.empty(by.shape[:-1] + (D,))
            c[..., 0::2] = by & 15
            c[..., 1::2] = by >> 4
        return (c - zp[phys].astype(np.float64)) * sc[phys].astype(np.float64)

    Ks, Vs = [], []
    for b in range(wl.batch):
        n = int(wl.seq_lens[b])
        Ks.append(deq(pool.kc, pool.ks, pool.kz, b, n))
        Vs.append(deq(pool.vc, pool.vs, pool.vz, b, n))
    q = W.bf16_bits_to_f32(wl.q_bits).astype(np.float64)
    ref = _dense_reference(q, Ks, Vs, wl.softmax_scale, wl.num_kv_heads)
    np.testing.assert_allclose(out.reshape(ref.shape), ref, rtol=1e-12, atol=1e-12)
    # and the quantised attention stays close to the bf16 one
    kv = [_seq_kv(wl, b) for b in range(wl.batch)]
    ref16 = _dense_reference(q, [k for k, _ in kv], [v for _, v in kv], wl.softmax_scale,
                             wl.num_kv_heads)
    tol = 0.05 if dt == "uint8" else 0.6
    assert np.abs(out.reshape(ref.shape) - ref16).max() < tol


def _pool_with(kv_rows_k, kv_rows_v, bs=16, D=8, Hkv=1, scale=1.0, perm_seed=0):
    """One sequence whose tokens are given explicitly; returns (pool, table, seq_lens)."""
    n = kv_rows_k.shape[0]
    nb = -(-n // bs)
    P = nb + 2
    table = np.full((1, nb), -1, np.int32)
    table[0] = np.random.default_rng(perm_seed).permutation(P)[:nb]
    pool = oracle.OraclePool("bf16", P, Hkv, bs, D, fill=0x7FC0)
    st = pool.append(kv_rows_k, kv_rows_v, np.array([0, n], np.int32), np.array([0], np.int32), table)
    assert st == 0
    return pool, table, np.array([n], np.int32)


def test_single_token_gives_v0():
    rng = np.random.default_rng(1)
    k = W.f32_to_bf16_bits(rng.normal(0, 1, (1, 1, 8)).astype(np.float32))
    v = W.f32_to_bf16_bits(rng.normal(0, 1, (1, 1, 8)).astype(np.float32))
    pool, table, sl = _pool_with(k, v)
    q = W.f32_to_bf16_bits(rng.normal(0, 1, (1, 3, 8)).astype(np.float32))
    out, st = pool.decode(q, table, sl, 0.3)
    assert st == 0
    for h in range(3):
        np.testing.assert_array_equal(out[h], W.bf16_bits_to_f32(v[0, 0]).astype(np.float64))


def test_identical_keys_give_mean_of_v():
    rng = np.random.default_rng(2)
    n = 37
    k = np.repeat(W.f32_to_bf16_bits(rng.normal(0, 1, (1, 1, 8)).astype(np.float32)), n, axis=0)
    v = W.f32_to_bf16_bits(rng.normal(0, 1, (n, 1, 8)).astype(np.float32))
    pool, table, sl = _pool_with(k, v)
    q = W.f32_to_bf16_bits(rng.normal(0, 1, (1, 2, 8)).astype(np.float32))
    out, st = pool.decode(q, table, sl, 0.5)
    mean = W.bf16_bits_to_f32(v[:, 0]).astype(np.float64).mean(axis=0)
    np.testing.assert_allclose(out[0], mean, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(out[1], mean, rtol=1e-13, atol=1e-14)


def test_hand_worked_two_token_softmax():
    """q = (1, 0), K0 = (0, 5), K1 = (1, -5), scale = ln 3: scores (0, ln 3),
    weights (1/4, 3/4); V0 = (1, 0), V1 = (0, 2) -> out = (0.25, 1.5)."""
    k = W.f32_to_bf16_bits(np.array([[[0, 5]], [[1, -5]]], np.float32))
    v = W.f32_to_bf16_bits(np.array([[[1, 0]], [[0, 2]]], np.float32))
    pool, table, sl = _pool_with(k, v, D=2)
    q = W.f32_to_bf16_bits(np.array([[[1, 0]]], np.float32))
    out, st = pool.decode(q, table, sl, math.log(3.0))
    np.testing.assert_allclose(out[0], [0.25, 1.5], rtol=1e-14)


def test_dominant_key_on_a_later_page_selects_its_value():
    """A key whose score exceeds every other by ~60 puts all weight on its
    value, wherever the page table places its block."""
    n, D = 45, 8
    rng = np.random.default_rng(3)
    kf = rng.normal(0, 0.1, (n, 1, D)).astype(np.float32)
    kf[33, 0, 0] = 64.0
    k = W.f32_to_bf16_bits(kf)
    v = W.f32_to_bf16_bits(rng.normal(0, 1, (n, 1, D)).astype(np.float32))
    q = W.f32_to_bf16_bits(np.array([[[1.0] + [0.0] * (D - 1)]], np.float32))
    for seed in range(3):
        pool, table, sl = _pool_with(k, v, D=D, perm_seed=seed)
        out, _ = pool.decode(q, table, sl, 1.0)
        np.testing.assert_allclose(out[0], W.bf16_bits_to_f32(v[33, 0]), rtol=1e-20, atol=1e-20)


def test_block_placement_permutation_invariance():
    wl = W.random_small(4, "uint8")
    pool = _load(wl)
    out, _ = pool.decode(wl.q_bits, wl.block_table, wl.seq_lens, wl.softmax_scale)
    # move every block to a new physical id (permute pool rows and tables alike)
    perm = np.random.default_rng(9).permutation(wl.num_blocks)
    inv = np.argsort(perm)
    moved = oracle.OraclePool("uint8", wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim)
    for name in ("kc", "vc", "ks", "vs", "kz", "vz"):
        getattr(moved, name)[...] = getattr(pool, name)[inv]
    table = np.where(wl.block_table >= 0, perm[np.maximum(wl.block_table, 0)], -1).astype(np.int32)
    out2, _ = moved.decode(wl.q_bits, table, wl.seq_lens, wl.softmax_scale)
    np.testing.assert_array_equal(out, out2)


def test_gqa_equals_mha_on_repeated_kv():
    """Grouped heads read KV head h // g: an MHA pool whose KV heads are the
    repeat_kv expansion gives identical outputs."""
    wl = W.random_small(8, "bf16")
    while wl.group_size == 1:
        wl = W.random_small(int(wl.q_bits.sum()) % 97 + 50, "bf16")
    g = wl.group_size
    pool = _load(wl)
    out, _ = pool.decode(wl.q_bits, wl.block_table, wl.seq_lens, wl.softmax_scale)
    mha = oracle.OraclePool("bf16", wl.num_blocks, wl.num_q_heads, wl.block_size, wl.head_dim)
    mha.k16[...] = np.repeat(pool.k16, g, axis=1)
    mha.v16[...] = np.repeat(pool.v16, g, axis=1)
    out2, _ = mha.decode(wl.q_bits, wl.block_table, wl.seq_lens, wl.softmax_scale)
    np.testing.assert_array_equal(out, out2)


def test_empty_sequence_gives_zero_row_and_bad_table_is_reported():
    wl = W.make_case("empty", 77, 2, 4, 2, 64, 16, "bf16", [0, 20])
    pool = _load(wl, leave_last=False)
    out, st = pool.decode(wl.q_bits, wl.block_table, wl.seq_lens, wl.softmax_scale)
    assert st == 0 and np.all(out[:4] == 0) and np.isfinite(out).all()
    bad = wl.block_table.copy()
    bad[1, 0] = wl.num_blocks
    _, st = pool.decode(wl.q_bits, bad, wl.seq_lens, wl.softmax_scale)
    assert st == -1


def test_row_subset_matches_full_decode():
    wl = W.random_small(2, "uint4")
    pool = _load(wl)
    full, _ = pool.decode(wl.q_bits, wl.block_table, wl.seq_lens, wl.softmax_scale)
    rows = np.array([wl.batch * wl.num_q_heads - 1, 0], np.int64)
    part, _ = pool.decode(wl.q_bits, wl.block_table, wl.seq_lens, wl.softmax_scale, rows=rows)
    np.testing.assert_array_equal(part, full[rows])


def test_prefix_sharing_layout_matches_private_copy():
    """Sequences that share prefix blocks attend exactly as if each held a
    private copy of its prefix."""
    wl = W.prefix_mix(seed=5, batch=16, n_groups=2, prefix_tokens=64, median=60, sigma=0.6,
                      max_len=200)
    pool = _load(wl)
    rows = np.arange(wl.batch * wl.num_q_heads, dtype=np.int64)
    out, st = pool.decode(wl.q_bits, wl.block_table, wl.seq_lens, wl.softmax_scale, rows)
    assert st == 0
    q = W.bf16_bits_to_f32(wl.q_bits).astype(np.float64)
    kv = [_seq_kv(wl, b) for b in range(wl.batch)]
    ref = _dense_reference(q, [k for k, _ in kv], [v for _, v in kv], wl.softmax_scale,
                           wl.num_kv_heads)
    np.testing.assert_allclose(out.reshape(ref.shape), ref, rtol=1e-12, atol=1e-12)
    assert (wl.shared_blocks > 0).any()
