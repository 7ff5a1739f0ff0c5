"""Pins for the oracle's KV quantiser and append (CPU only).

The quantiser follows the asymmetric per-channel formula of the heterogeneous
engine article (section 2.6) with the round-half-even / int32-zp / degenerate
readings; append follows the paged layout of the TFFInfer KVCache (section
3.6.4: page = token / PAGE_SIZE, slot = token % PAGE_SIZE) and the article's
per-block KV scales (section 2.4).
"""
import os

import numpy as np
import pytest

from oracle import oracle
from paged_gqa_decode_02_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "quant_pins.txt")


def _pins():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        L, vals, sc, zp, codes, what = [x.strip() for x in line.split("|")]
        rows.append((int(L), [float(v) for v in vals.split(",")], int(sc, 16), int(zp),
                     [int(c) for c in codes.split(",")], what))
    return rows


@pytest.mark.parametrize("pin", _pins(), ids=lambda p: p[5][:40])
def test_hand_worked_pins(pin):
    L, vals, scale_bits, zp, codes, _ = pin
    sc, z, c = oracle.quant_channel(vals, L)
    assert int(np.float32(sc).view(np.uint32)) == scale_bits
    assert z == zp
    assert list(c) == codes


def test_pin_file_has_all_cases():
    assert len(_pins()) == 9


@pytest.mark.parametrize("L", [255, 15])
def test_round_trip_bound_random_blocks(L):
    """|dequant - x| <= scale/2 when no clamp acted, else <= scale (the zero
    point's own rounding adds up to half a step), each plus the fp32 rounding
    of x / scale (at most 2^-23 |x|); codes stay in [0, L]; the
    block minimum and maximum map to codes 0 and L (up to fp32 rounding)."""
    rng = np.random.default_rng(7)
    for trial in range(400):
        n = int(rng.integers(2, 33))
        off = rng.normal(0, 3)
        vals = (rng.normal(off, rng.uniform(0.01, 5), n)).astype(np.float32)
        vals = W.bf16_bits_to_f32(W.f32_to_bf16_bits(vals))
        sc, zp, codes = oracle.quant_channel(vals, L)
        assert sc > 0
        assert codes.min() >= 0 and codes.max() <= L
        deq = (codes.astype(np.float64) - zp) * np.float64(sc)
        err = np.abs(deq - vals.astype(np.float64))
        raw = np.rint(vals.astype(np.float64) / np.float64(sc)) + zp
        unclamped = (raw >= 0) & (raw <= L)
        slack = 2.0 ** -22 * np.abs(vals.astype(np.float64))
        assert np.all(err[unclamped] <= 0.5 * sc + slack[unclamped])
        assert np.all(err <= 1.0 * sc + slack)
        assert codes[np.argmin(vals)] <= 1
        assert codes[np.argmax(vals)] >= L - 1


@pytest.mark.parametrize("L", [255, 15])
def test_degenerate_blocks_round_trip_exactly(L):
    for v in [0.75, -0.75, 3.0, -1e-3, 12345.0, 0.0]:
        for n in (1, 5):
            sc, zp, codes = oracle.quant_channel([v] * n, L)
            assert np.all(codes == 0)
            assert np.float32(np.float32(0 - zp) * np.float32(sc)) == np.float32(v)


def _gather_tokens(pool_arr, table, b, n, bs):
    """Independent restatement of the addressing rule: token t of sequence b
    sits in slot t % bs of physical block table[b][t // bs]."""
    t = np.arange(n)
    return pool_arr[table[b, t // bs], :, t % bs]


def test_bf16_append_is_an_exact_scatter():
    wl = W.random_small(3, "bf16")
    pool = oracle.OraclePool("bf16", wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim,
                             fill=0x7FC0)
    for call in wl.fill_calls(leave_last=True) + [wl.step_call()]:
        assert pool.append_call(call) == 0
    for b in range(wl.batch):
        n = int(wl.seq_lens[b])
        o = int(wl.tok_off[b])
        np.testing.assert_array_equal(_gather_tokens(pool.k16, wl.block_table, b, n, wl.block_size),
                                      wl.k_bits[o:o + n])
        np.testing.assert_array_equal(_gather_tokens(pool.v16, wl.block_table, b, n, wl.block_size),
                                      wl.v_bits[o:o + n])


@pytest.mark.parametrize("dt", ["uint8", "uint4"])
def test_bulk_quant_append_matches_per_channel_quantiser(dt):
    wl = W.random_small(11, dt)
    L = 255 if dt == "uint8" else 15
    pool = oracle.OraclePool(dt, wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim)
    assert pool.append_call(wl.fill_calls(leave_last=False)[0]) == 0
    bs, D = wl.block_size, wl.head_dim
    for b in range(wl.batch):
        n = int(wl.seq_lens[b])
        o = int(wl.tok_off[b])
        kv = W.bf16_bits_to_f32(wl.k_bits[o:o + n])  # [n, Hkv, D]
        for blk in range(-(-n // bs)):
            phys = wl.block_table[b, blk]
            toks = kv[blk * bs: min(n, (blk + 1) * bs)]
            for h in range(wl.num_kv_heads):
                for c in (0, 1, D // 2, D - 1):
                    sc, zp, codes = oracle.quant_channel(toks[:, h, c], L)
                    assert pool.ks[phys, h, c] == sc and pool.kz[phys, h, c] == zp
                    if dt == "uint8":
                        got = pool.kc[phys, h, :len(toks), c]
                    else:
                        byte = pool.kc[phys, h, :len(toks), c // 2]
                        got = (byte >> 4) if c % 2 else (byte & 15)
                    np.testing.assert_array_equal(got, codes)


def test_uint4_nibble_order():
    """Channel 2j goes to the low nibble, 2j+1 to the high nibble. Channel 0
    holds the uint4 pin (-1, 0, 1) -> codes 0, 7, 14; channel 1 is that
    column negated (1, 0, -1) -> codes 14, 7, 0."""
    D, bs = 2, 16
    pool = oracle.OraclePool("uint4", 1, 1, bs, D)
    vals = np.array([[-1.0, 1.0], [0.0, 0.0], [1.0, -1.0]], np.float32)
    bits = W.f32_to_bf16_bits(vals).reshape(3, 1, D)
    st = pool.append(bits, bits, np.array([0, 3], np.int32), np.array([0], np.int32),
                     np.array([[0]], np.int32))
    assert st == 0
    assert list(pool.kc[0, 0, :3, 0]) == [0 | (14 << 4), 7 | (7 << 4), 14 | (0 << 4)]


@pytest.mark.parametrize("dt", ["uint8", "uint4"])
def test_tail_block_requantises_old_values(dt):
    """Appending into a partly filled block re-quantises it from the
    dequantised stored values (fp32 (code - zp) * scale) plus the new bf16
    values."""
    L = 255 if dt == "uint8" else 15
    D, bs, Hkv = 4, 16, 1
    rng = np.random.default_rng(5)
    first = W.f32_to_bf16_bits(rng.normal(0, 1, (5, Hkv, D)).astype(np.float32))
    new = W.f32_to_bf16_bits(rng.normal(0, 3, (2, Hkv, D)).astype(np.float32))
    pool = oracle.OraclePool(dt, 2, Hkv, bs, D)
    table = np.array([[1, 0]], np.int32)
    assert pool.append(first, first, np.array([0, 5], np.int32), np.array([0], np.int32), table) == 0
    sc0, zp0 = pool.ks[1, 0].copy(), pool.kz[1, 0].copy()
    if dt == "uint8":
        codes0 = pool.kc[1, 0, :5].astype(np.int32)
    else:
        by = pool.kc[1, 0, :5]
        codes0 = np.stack([by[:, c // 2] >> 4 if c % 2 else by[:, c // 2] & 15 for c in range(D)], 1)
    old_vals = ((codes0 - zp0[None, :]).astype(np.float32) * sc0[None, :]).astype(np.float32)
    assert pool.append(new, new, np.array([0, 2], np.int32), np.array([5], np.int32), table) == 0
    for c in range(D):
        vals = np.concatenate([old_vals[:, c], W.bf16_bits_to_f32(new[:, 0, c])])
        sc, zp, codes = oracle.quant_channel(vals, L)
        assert pool.ks[1, 0, c] == sc and pool.kz[1, 0, c] == zp


def test_append_rejects_bad_table_entries():
    pool = oracle.OraclePool("uint8", 2, 1, 16, 4)
    bits = np.zeros((1, 1, 4), np.uint16)
    assert pool.append(bits, bits, np.array([0, 1], np.int32), np.array([0], np.int32),
                       np.array([[2]], np.int32)) == -1
    assert pool.append(bits, bits, np.array([0, 1], np.int32), np.array([16], np.int32),
                       np.array([[0]], np.int32)) == -1
