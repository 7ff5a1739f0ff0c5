"""The host block manager's CPU swap tier driving real page moves: a
sequence's blocks go to a pinned host buffer (pa_swap_blocks), other
sequences reuse and overwrite the freed GPU blocks, and the sequence comes
back into fresh blocks. The pool stays bit-exact with the oracle fed the same
tables and block moves, and the attention matches it."""
import numpy as np
import pytest

from oracle import oracle
from paged_gqa_decode_02_gb300 import binding as B
from paged_gqa_decode_02_gb300 import workloads as W
from tests import harness as H
from tests.test_gpu_block_manager import _kv_for

pytestmark = pytest.mark.gpu

_NAMES = ("k16", "v16", "kc", "vc", "ks", "vs", "kz", "vz")


@pytest.mark.parametrize("dt", ["bf16", "uint8", "uint4", "fp8"])
def test_swap_out_reuse_and_swap_in(dt):
    torch = H.torch_mod()
    bs, Hkv, Hq, D, nb, MB = 16, 2, 8, 128, 12, 12
    rng = np.random.default_rng(21)
    bm = B.BlockManager(nb, bs)
    bm.set_cpu_blocks(6)
    g, o = H.make_pools(W.make_case("swap", 21, 1, Hq, Hkv, D, bs, dt, [1], extra_blocks=nb - 1))
    host = torch.zeros(6 * g.block_bytes(), dtype=torch.uint8).pin_memory()
    o_host = {}  # oracle side of the host tier: slot -> arrays of one block
    toks = {}

    def admit(sid, tokens):
        cached = bm.add_sequence(sid, tokens)
        table, _ = bm.block_table(sid, MB)
        k, v = _kv_for(tokens, Hkv, D)
        n_new = len(tokens) - cached
        args = (k[cached:], v[cached:], np.array([0, n_new], np.int32), np.array([cached], np.int32), table[None, :])
        g.append_kv(*(H.dev(a) for a in args), max_new_per_seq=n_new)
        assert o.append(*args) == 0
        toks[sid] = list(tokens)

    def swap_out(sid):
        moves = bm.swap_out(sid)
        g.swap_blocks(host, [b for b, _ in moves], [s for _, s in moves], "out")
        for b, s in moves:
            o_host[s] = {n: getattr(o, n)[b].copy() for n in _NAMES if getattr(o, n) is not None}
        return moves

    def swap_in(sid):
        moves = bm.swap_in(sid)
        g.swap_blocks(host, [b for _, b in moves], [s for s, _ in moves], "in")
        for s, b in moves:
            for n, a in o_host.pop(s).items():
                getattr(o, n)[b] = a
        return moves

    admit(1, [int(x) for x in rng.integers(0, 50, 45)])   # 3 blocks
    admit(2, [int(x) for x in rng.integers(50, 99, 20)])  # 2 blocks
    out1 = swap_out(1)
    assert len(out1) == 3
    torch.cuda.synchronize()
    # another sequence takes (and overwrites) every free block, sequence 1's included
    admit(3, [int(x) for x in rng.integers(100, 150, 16 * 10)])
    assert bm.num_free_blocks() == 0
    bm.free_sequence(3)
    back = swap_in(1)
    assert len(back) == 3
    torch.cuda.synchronize()
    H.assert_pools_equal(g, o)

    sids = [1, 2]
    table = np.stack([bm.block_table(s, MB)[0] for s in sids]).astype(np.int32)
    lens = np.array([len(toks[s]) for s in sids], np.int32)
    q = W.f32_to_bf16_bits(rng.standard_normal((len(sids), Hq, D)).astype(np.float32))
    scale = 1.0 / np.sqrt(D)
    ref, st = o.decode(q, table, lens, scale)
    assert st == 0
    # and the same attention as a fresh oracle pool holding sequence 1's tokens directly
    fresh = oracle.OraclePool(dt, nb, Hkv, bs, D)
    k, v = _kv_for(toks[1], Hkv, D)
    assert fresh.append(k, v, np.array([0, 45], np.int32), np.array([0], np.int32), table[:1]) == 0
    ref1, _ = fresh.decode(q[:1], table[:1], lens[:1], scale)
    np.testing.assert_array_equal(ref[:Hq], ref1)
    out = g.decode(H.dev(q), H.dev(table), H.dev(lens), scale)
    H.check_attention(out.cpu().numpy().reshape(-1, D), ref, f"swap {dt}")
    assert g.device_error() == (0, 0)
    g.close()


def test_swap_blocks_validates_before_copying():
    torch = H.torch_mod()
    g = B.PagedKVPool(4, 16, 2, 64, "bf16")
    host = torch.zeros(2 * g.block_bytes(), dtype=torch.uint8)
    assert g.block_bytes() == 2 * 2 * 16 * 64 * 2
    for blocks, slots in (([4], [0]), ([0], [2]), ([-1], [0])):
        with pytest.raises(B.PagedAttnError) as e:
            g.swap_blocks(host, blocks, slots, "out")
        assert e.value.status == 1
    g.close()
