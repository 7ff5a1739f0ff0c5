"""Pins for the oracle's multi-token query attention (CPU only).

Several query tokens per sequence (a chunk of a prefill, or the draft tokens
a speculative step verifies: the engine article, sections 2.2 and 4.2, mixes
prefill chunks into decode steps; TFFInfer, section 9.3, plans speculative
decoding). All n_q new tokens are stored before the call, and query token i
attends causally to the first seq_len - (n_q - 1 - i) tokens. The tests pin
the oracle to an independent dense causal attention written with numpy, to
closed forms, and to the causal cut itself.
"""
import numpy as np
import pytest

from oracle import oracle
from paged_gqa_decode_02_gb300 import workloads as W


def _load(wl):
    pool = oracle.OraclePool(wl.kv_dtype, wl.num_blocks, wl.num_kv_heads, wl.block_size,
                             wl.head_dim, fill=0x7FC0 if wl.kv_dtype == "bf16" else 0)
    for c in wl.fill_calls(leave_last=False):
        assert pool.append_call(c) == 0
    return pool


def _queries(seed, B, n_q, Hq, D):
    rng = np.random.default_rng([seed, 11])
    return W.f32_to_bf16_bits(rng.standard_normal((B, n_q, Hq, D), dtype=np.float32))


def _gathered_kv(pool, wl, b):
    """Dequantised K, V [n, Hkv, D] of sequence b, gathered in numpy."""
    bs, D = wl.block_size, wl.head_dim
    n = int(wl.seq_lens[b])
    t = np.arange(n)
    phys = wl.block_table[b, t // bs]
    if wl.kv_dtype == "bf16":
        return (W.bf16_bits_to_f32(pool.k16[phys, :, t % bs, :]).astype(np.float64),
                W.bf16_bits_to_f32(pool.v16[phys, :, t % bs, :]).astype(np.float64))
    out = []
    for codes, sc, zp in ((pool.kc, pool.ks, pool.kz), (pool.vc, pool.vs, pool.vz)):
        if wl.kv_dtype == "uint8":
            c = codes[phys, :, t % bs, :].astype(np.float64)
        else:
            by = codes[phys, :, t % bs, :]
            c = np.empty(by.shape[:-1] + (D,))
            c[..., 0::2] = by & 15
            c[..., 1::2] = by >> 4
        out.append((c - zp[phys].astype(np.float64)) * sc[phys].astype(np.float64))
    return out[0], out[1]


def _dense_causal(q, K, V, scale, Hkv):
    """softmax(q K^T * scale + causal mask) V for one sequence: q [n_q, Hq, D],
    K/V [n, Hkv, D]; query i sits at position n - n_q + i."""
    n_q, Hq, D = q.shape
    n = K.shape[0]
    g = Hq // Hkv
    Kx = np.repeat(K, g, axis=1).transpose(1, 0, 2)  # [Hq, n, D]
    Vx = np.repeat(V, g, axis=1).transpose(1, 0, 2)
    s = np.einsum("ihd,hnd->ihn", q, Kx) * scale  # [n_q, Hq, n]
    pos = n - n_q + np.arange(n_q)
    mask = np.arange(n)[None, :] <= pos[:, None]  # [n_q, n]
    out = np.zeros((n_q, Hq, D))
    for i in range(n_q):
        if not mask[i].any():
            continue
        si = np.where(mask[i][None, :], s[i], -np.inf)
        si = si - si.max(axis=1, keepdims=True)
        p = np.exp(si)
        p /= p.sum(axis=1, keepdims=True)
        out[i] = np.einsum("hn,hnd->hd", p, Vx)
    return out


@pytest.mark.parametrize("dt", ["bf16", "uint8", "uint4"])
@pytest.mark.parametrize("n_q", [1, 2, 5])
def test_matches_dense_causal_attention(dt, n_q):
    wl = W.make_case(f"mq_{dt}", 31 + n_q, 3, 8, 2, 64, 16, dt, [40, n_q, 17], extra_blocks=1,
                     channel_offset_sigma=None if dt == "bf16" else 0.5)
    pool = _load(wl)
    q = _queries(5, wl.batch, n_q, wl.num_q_heads, wl.head_dim)
    out, st = pool.decode_multi(q, wl.block_table, wl.seq_lens, wl.softmax_scale)
    assert st == 0
    out = out.reshape(wl.batch, n_q, wl.num_q_heads, wl.head_dim)
    qf = W.bf16_bits_to_f32(q).astype(np.float64)
    for b in range(wl.batch):
        K, V = _gathered_kv(pool, wl, b)
        ref = _dense_causal(qf[b], K, V, wl.softmax_scale, wl.num_kv_heads)
        np.testing.assert_allclose(out[b], ref, rtol=1e-12, atol=1e-12)


def test_first_token_of_a_fresh_sequence_sees_only_itself():
    """seq_len == n_q (nothing cached before the chunk): query 0 attends to
    token 0 alone, so its output is V_0 exactly; query i sees i + 1 tokens."""
    n_q = 4
    wl = W.make_case("mq_fresh", 41, 1, 4, 1, 64, 16, "bf16", [n_q])
    pool = _load(wl)
    q = _queries(6, 1, n_q, 4, 64)
    out, st = pool.decode_multi(q, wl.block_table, wl.seq_lens, wl.softmax_scale)
    assert st == 0
    v0 = W.bf16_bits_to_f32(wl.v_bits[0, 0]).astype(np.float64)
    for h in range(4):
        np.testing.assert_array_equal(out[h], v0)
    assert not np.allclose(out[4], v0)  # query 1 also sees token 1


def test_identical_keys_give_prefix_means():
    """With one key repeated, query i weights its visible tokens equally and
    returns the mean of V over them."""
    n, n_q, D = 37, 6, 8
    rng = np.random.default_rng(4)
    k = np.repeat(W.f32_to_bf16_bits(rng.normal(0, 1, (1, 1, D)).astype(np.float32)), n, axis=0)
    v = W.f32_to_bf16_bits(rng.normal(0, 1, (n, 1, D)).astype(np.float32))
    pool = oracle.OraclePool("bf16", 4, 1, 16, D)
    table = np.array([[2, 0, 3]], np.int32)
    assert pool.append(k, v, np.array([0, n], np.int32), np.array([0], np.int32), table) == 0
    q = W.f32_to_bf16_bits(rng.normal(0, 1, (1, n_q, 2, D)).astype(np.float32))
    out, st = pool.decode_multi(q, table, np.array([n], np.int32), 0.7)
    assert st == 0
    vf = W.bf16_bits_to_f32(v[:, 0]).astype(np.float64)
    for i in range(n_q):
        mean = vf[: n - n_q + i + 1].mean(axis=0)
        for h in range(2):
            np.testing.assert_allclose(out[i * 2 + h], mean, rtol=1e-13, atol=1e-14)


def test_later_tokens_do_not_reach_earlier_queries():
    """Changing the K/V of the last token changes only the last query's row."""
    n_q = 3
    wl = W.make_case("mq_cut", 42, 1, 2, 1, 64, 16, "bf16", [30])
    pool = _load(wl)
    q = _queries(7, 1, n_q, 2, 64)
    out, _ = pool.decode_multi(q, wl.block_table, wl.seq_lens, wl.softmax_scale)
    last = wl.block_table[0, 29 // 16]
    pool.k16[last, 0, 29 % 16] ^= 0x0040
    pool.v16[last, 0, 29 % 16] ^= 0x0040
    out2, _ = pool.decode_multi(q, wl.block_table, wl.seq_lens, wl.softmax_scale)
    np.testing.assert_array_equal(out[:4], out2[:4])
    assert not np.array_equal(out[4:], out2[4:])


def test_single_query_token_is_the_decode_step():
    wl = W.random_small(3, "uint8")
    pool = _load(wl)
    a, _ = pool.decode(wl.q_bits, wl.block_table, wl.seq_lens, wl.softmax_scale)
    b, _ = pool.decode_multi(wl.q_bits[:, None], wl.block_table, wl.seq_lens, wl.softmax_scale)
    np.testing.assert_array_equal(a, b)


def test_queries_before_the_first_token_give_zero_rows_and_bad_tables_are_reported():
    """A sequence shorter than the chunk (reading: its leading queries see no
    token) gives zero rows there; an out-of-range table entry is reported."""
    wl = W.make_case("mq_short", 43, 2, 2, 1, 64, 16, "bf16", [2, 20])
    pool = _load(wl)
    q = _queries(8, 2, 4, 2, 64)
    out, st = pool.decode_multi(q, wl.block_table, wl.seq_lens, wl.softmax_scale)
    assert st == 0
    assert np.all(out[:4] == 0) and np.all(np.abs(out[4:8]).sum(axis=1) > 0)
    bad = wl.block_table.copy()
    bad[1, 1] = wl.num_blocks
    _, st = pool.decode_multi(q, bad, wl.seq_lens, wl.softmax_scale)
    assert st == -1


def test_row_subset_matches_all_rows():
    wl = W.make_case("mq_rows", 44, 2, 4, 2, 64, 32, "uint4", [50, 9], channel_offset_sigma=0.5)
    pool = _load(wl)
    q = _queries(9, 2, 3, 4, 64)
    full, _ = pool.decode_multi(q, wl.block_table, wl.seq_lens, wl.softmax_scale)
    rows = np.array([23, 0, 13], np.int64)
    part, _ = pool.decode_multi(q, wl.block_table, wl.seq_lens, wl.softmax_scale, rows=rows)
    np.testing.assert_array_equal(part, full[rows])
