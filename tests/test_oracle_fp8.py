"""Pins for the oracle's fp8 (E4M3) KV format (CPU only).

The encoding is the E4M3 format of the OCP 8-bit floating point
specification, rounded to nearest-even and saturated to +-448. The pages fix
no FP8 scheme (TFFInfer, section 9.3, lists FP8 among the quantisation formats
to add), so the scale follows the integer formats' granularity: one
symmetric scale max|x| / 448 per (block, kv head, channel). These tests pin
the oracle to hand-worked values, to PyTorch's own float8_e4m3fn conversion
(a library routine) over every code and every rounding boundary, to a
round-trip bound, and to an independent dense attention over codes decoded
by PyTorch.
"""
import math
import os

import numpy as np
import pytest

from oracle import oracle
from paged_gqa_decode_02_gb300 import workloads as W

torch = pytest.importorskip("torch")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "fp8_pins.txt")


def _rows(kind):
    out = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        f = [x.strip() for x in line.split("|")]
        if f[0] == kind:
            out.append(f[1:])
    return out


def _torch_value(codes):
    """float64 values of E4M3 bit patterns through PyTorch's float8 type."""
    c = torch.from_numpy(np.asarray(codes, np.uint8).copy())
    return c.view(torch.float8_e4m3fn).to(torch.float32).numpy().astype(np.float64)


def _torch_encode(y):
    """PyTorch's float32 -> float8_e4m3fn conversion (finite, |y| <= 448)."""
    t = torch.from_numpy(np.ascontiguousarray(y, np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _all_finite_values():
    v = _torch_value(np.arange(256))
    return np.unique(v[np.isfinite(v)])


@pytest.mark.parametrize("row", _rows("encode"), ids=lambda r: r[2][:40])
def test_hand_worked_encodings(row):
    x, code, _ = row
    got = int(oracle.e4m3_encode(np.array([float(x)], np.float32))[0])
    assert got == int(code, 16), f"{x}: {got:#x}"


@pytest.mark.parametrize("row", _rows("value"), ids=lambda r: r[2][:40])
def test_hand_worked_values(row):
    code, value, _ = row
    got = oracle.e4m3_value([int(code, 16)])[0]
    if value == "nan":
        assert math.isnan(got)
    else:
        assert got == float(value)


@pytest.mark.parametrize("row", _rows("channel"), ids=lambda r: r[3][:40])
def test_hand_worked_channels(row):
    vals, scale_bits, codes, _ = row
    sc, c = oracle.quant_channel_fp8([float(v) for v in vals.split(",")])
    assert int(np.float32(sc).view(np.uint32)) == int(scale_bits, 16)
    assert [int(x) for x in c] == [int(x, 16) for x in codes.split(",")]


def test_pin_file_has_all_cases():
    assert (len(_rows("encode")), len(_rows("value")), len(_rows("channel"))) == (20, 8, 6)


def test_every_code_decodes_like_pytorch():
    ours = oracle.e4m3_value(np.arange(256))
    ref = _torch_value(np.arange(256))
    assert np.array_equal(np.isnan(ours), np.isnan(ref)) and np.isnan(ours).sum() == 2
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    assert np.array_equal(np.signbit(ours[ok]), np.signbit(ref[ok]))


def test_every_finite_value_encodes_back_to_its_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = oracle.e4m3_value(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)


def test_rounding_boundaries_match_pytorch():
    """Every midpoint between neighbouring finite values (the ties) and the
    float32 neighbours on either side of it, positive and negative."""
    v = _all_finite_values()
    v = v[v >= 0]
    mids = ((v[:-1] + v[1:]) / 2).astype(np.float32)  # exact: the spacing is a power of two
    ys = np.concatenate([mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9)),
                         v.astype(np.float32)])
    ys = ys[np.abs(ys) <= 448]
    ys = np.concatenate([ys, -ys])
    assert np.array_equal(oracle.e4m3_encode(ys), _torch_encode(ys))


def test_random_values_across_binades_match_pytorch():
    rng = np.random.default_rng(3)
    ys = (rng.uniform(-1, 1, 20000) * np.exp2(rng.uniform(-14, 8.8, 20000))).astype(np.float32)
    ys = ys[np.abs(ys) <= 448]
    assert np.array_equal(oracle.e4m3_encode(ys), _torch_encode(ys))


def test_round_trip_bound_random_blocks():
    """|value(code) * scale - x| is at most half a spacing of E4M3 at x / scale
    (2^-4 relative for normals, 2^-10 absolute below 2^-6), scaled, plus the
    fp32 rounding of x / scale; the largest magnitude maps to +-448."""
    rng = np.random.default_rng(8)
    for trial in range(300):
        n = int(rng.integers(1, 33))
        vals = rng.normal(rng.normal(0, 2), rng.uniform(0.01, 5), n).astype(np.float32)
        vals = W.bf16_bits_to_f32(W.f32_to_bf16_bits(vals))
        sc, codes = oracle.quant_channel_fp8(vals)
        assert sc > 0
        deq = _torch_value(codes.astype(np.uint8)) * np.float64(sc)
        y = vals.astype(np.float64) / np.float64(sc)
        half = np.where(np.abs(y) >= 2.0 ** -6, np.abs(y) * 2.0 ** -4, 2.0 ** -10)
        bound = (half * (1 + 2.0 ** -20) + np.abs(y) * 2.0 ** -23) * np.float64(sc)
        assert np.all(np.abs(deq - vals) <= bound), trial
        i = int(np.argmax(np.abs(vals)))
        assert abs(_torch_value([codes[i]])[0]) == 448.0


def _fp8_pool_case(seed, bs=16, D=64, Hkv=2, g=2, lens=(37, 5, 16)):
    wl = W.make_case(f"fp8_{seed}", seed, len(lens), Hkv * g, Hkv, D, bs, "fp8", list(lens),
                     extra_blocks=2, channel_offset_sigma=0.5)
    pool = oracle.OraclePool("fp8", wl.num_blocks, wl.num_kv_heads, bs, D)
    for c in wl.fill_calls(leave_last=True) + [wl.step_call()]:
        assert pool.append_call(c) == 0
    return wl, pool


def test_pool_holds_no_zero_points_and_codes_use_the_byte_layout():
    wl, pool = _fp8_pool_case(1)
    assert pool.kz is None and pool.vz is None
    assert pool.kc.shape == (wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim)


def test_bulk_append_stores_the_channel_quantiser_codes():
    """A bulk load quantises each (block, kv head, channel) once from the bf16
    values: the pool holds exactly the channel quantiser's scale and codes."""
    wl = W.make_case("fp8_bulk", 4, 2, 4, 2, 64, 16, "fp8", [40, 9], extra_blocks=1)
    pool = oracle.OraclePool("fp8", wl.num_blocks, 2, 16, 64)
    for c in wl.fill_calls(leave_last=False):
        assert pool.append_call(c) == 0
    k = W.bf16_bits_to_f32(wl.k_bits)
    for b in range(2):
        n = int(wl.seq_lens[b])
        for blk in range(-(-n // 16)):
            phys = wl.block_table[b, blk]
            t0, t1 = blk * 16, min(n, blk * 16 + 16)
            for h in range(2):
                for c in (0, 17, 63):
                    sc, codes = oracle.quant_channel_fp8(k[wl.tok_off[b] + t0: wl.tok_off[b] + t1, h, c])
                    assert pool.ks[phys, h, c] == sc
                    assert list(pool.kc[phys, h, : t1 - t0, c]) == list(codes)


def test_append_into_a_partial_block_requantises_from_stored_values():
    """Token 0 = 2.0 is stored alone (code 448 at scale 2/448); appending
    -1.0 re-quantises the block from float(448) * scale and the new value:
    the old code is 448 again and -1.0 lands on -224."""
    D, bs = 8, 16
    pool = oracle.OraclePool("fp8", 2, 1, bs, D)
    table = np.array([[1]], np.int32)
    two = W.f32_to_bf16_bits(np.full((1, 1, D), 2.0, np.float32))
    neg = W.f32_to_bf16_bits(np.full((1, 1, D), -1.0, np.float32))
    assert pool.append(two, two, np.array([0, 1], np.int32), np.array([0], np.int32), table) == 0
    assert np.all(pool.kc[1, 0, 0] == 0x7E)
    assert pool.append(neg, neg, np.array([0, 1], np.int32), np.array([1], np.int32), table) == 0
    assert np.all(pool.kc[1, 0, 0] == 0x7E) and np.all(pool.kc[1, 0, 1] == 0xF6)
    s_old = np.float32(448.0) * np.float32(np.float32(2.0) / np.float32(448.0))
    assert np.all(pool.ks[1, 0] == np.float32(s_old) / np.float32(448.0))


def _dense(q, K, V, scale):
    s = q @ K.T * scale
    s -= s.max()
    p = np.exp(s)
    return (p / p.sum()) @ V


def test_decode_matches_dense_attention_on_pytorch_decoded_codes():
    wl, pool = _fp8_pool_case(2)
    out, st = pool.decode(wl.q_bits, wl.block_table, wl.seq_lens, wl.softmax_scale)
    assert st == 0
    bs, g = wl.block_size, wl.group_size
    q = W.bf16_bits_to_f32(wl.q_bits).astype(np.float64)
    k16 = W.bf16_bits_to_f32(wl.k_bits).astype(np.float64)
    i = 0
    for b in range(wl.batch):
        n = int(wl.seq_lens[b])
        t = np.arange(n)
        phys = wl.block_table[b, t // bs]
        for h in range(wl.num_q_heads):
            j = h // g
            K = _torch_value(pool.kc[phys, j, t % bs, :]) * pool.ks[phys, j, :].astype(np.float64)
            V = _torch_value(pool.vc[phys, j, t % bs, :]) * pool.vs[phys, j, :].astype(np.float64)
            ref = _dense(q[b, h], K, V, wl.softmax_scale)
            np.testing.assert_allclose(out[i], ref, rtol=1e-12, atol=1e-12)
            # and the fp8 cache stays close to the bf16 one it was made from
            # (half a spacing, 2^-4 relative, per quantisation; the tail
            # block was quantised twice)
            Kb = k16[wl.tok_off[b]: wl.tok_off[b] + n, j]
            assert np.abs(K - Kb).max() <= 2 * 2.0 ** -4 * np.abs(Kb).max() * 1.01
            i += 1
