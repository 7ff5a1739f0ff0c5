"""GPU parity of the fused decode step (pa_decode_step): one decode launch
stores every sequence's new token (the thread block that reads the
sequence's last page re-quantises that block first) and attends. It must
leave the pool exactly as the oracle's append of one token per sequence does
(codes, scales and zero points bit for bit) and give the attention of the
oracle's decode after that append, for every KV format, split counts from one
slice to many slices per sequence, with and without the early plan, over
consecutive steps that cross block boundaries, and on the full-size
workloads."""
import numpy as np
import pytest

from paged_gqa_decode_02_gb300 import workloads as W
from tests import harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_gqa_decode_02_gb300 import build
    build.build()


def _rows(wl, call):
    """k_new / v_new [B, Hkv, D] of one token per sequence from an append call
    (rows of empty sequences stay zero)."""
    B, Hkv, D = wl.batch, wl.num_kv_heads, wl.head_dim
    k = np.zeros((B, Hkv, D), np.uint16)
    v = np.zeros((B, Hkv, D), np.uint16)
    for b in range(B):
        if call.cu_new[b + 1] > call.cu_new[b]:
            k[b] = call.k_bits[call.cu_new[b]]
            v[b] = call.v_bits[call.cu_new[b]]
    return k, v


def _step(g, wl, k, v, lens, splits, path="auto", early=False):
    torch = H.torch_mod()
    g.set_decode_path(path, early_plan=early)
    out = torch.full((wl.batch, wl.num_q_heads, wl.head_dim), float("nan"), dtype=torch.float32, device="cuda")
    g.decode_step(H.dev(k), H.dev(v), H.dev(wl.q_bits), H.dev(wl.block_table), H.dev(lens), wl.softmax_scale,
                  out=out, num_splits=splits)
    torch.cuda.synchronize()
    return out.cpu().numpy().reshape(wl.batch * wl.num_q_heads, wl.head_dim)


def _paths(dt, D):
    return ["cuda_core", "tensor_core"] if dt == "bf16" or D == 128 else ["cuda_core"]


@pytest.mark.parametrize("dt", ["bf16", "uint8", "uint4", "fp8"])
@pytest.mark.parametrize("seed", [1, 2, 3])
def test_step_matches_append_then_decode(dt, seed):
    base = W.random_small(40 + seed, dt)
    for path in _paths(dt, base.head_dim):
        for splits, early in ((0, True), (1, False), (7, False), (300, True)):
            wl = W.random_small(40 + seed, dt)
            g, o = H.load_both(wl, leave_last=True)
            call = wl.step_call()
            k, v = _rows(wl, call)
            got = _step(g, wl, k, v, wl.seq_lens, splits, path, early)
            assert o.append_call(call) == 0
            H.assert_pools_equal(g, o)
            ref, st = o.decode(wl.q_bits, wl.block_table, wl.seq_lens, wl.softmax_scale)
            assert st == 0
            H.check_attention(got, ref, f"{wl.name} {path} splits={splits} early={early}")
            assert g.device_error() == (0, 0)
            g.close()


@pytest.mark.parametrize("dt", ["bf16", "uint8", "uint4", "fp8"])
def test_consecutive_steps_cross_block_boundaries(dt):
    """Three steps in a row, each one token per sequence, lengths chosen so
    that new tokens land at the end of a block, at the start of a fresh block
    and inside one; an empty sequence stays empty."""
    bs = 16
    seq = [bs - 2, 2 * bs - 1, 0, bs + 5, 1]
    final = [n + 3 if n else 0 for n in seq]
    wl = W.make_case(f"steps_{dt}", 77, len(seq), 8, 2, 128, bs, dt, final, extra_blocks=2,
                     channel_offset_sigma=0.5 if dt != "bf16" else None)
    g, o = H.make_pools(wl)
    # load all but the last three tokens of every non-empty sequence
    for c in W.Workload.fill_calls(_truncated(wl, 3), leave_last=False):
        H.gpu_append(g, c)
        assert o.append_call(c) == 0
    for t in range(3, 0, -1):
        lens = np.array([n - t + 1 if n else 0 for n in final], np.int32)
        call = _token_call(wl, lens)
        k, v = _rows(wl, call)
        got = _step(g, wl, k, v, lens, 0, early=(t == 2))
        assert o.append_call(call) == 0
        H.assert_pools_equal(g, o)
        ref, st = o.decode(wl.q_bits, wl.block_table, lens, wl.softmax_scale)
        assert st == 0
        H.check_attention(got, ref, f"step {3 - t} {dt}")
    assert g.device_error() == (0, 0)
    g.close()


def _truncated(wl, drop):
    """The workload with every non-empty sequence `drop` tokens shorter (same
    tables and token values)."""
    import dataclasses
    lens = np.array([max(int(n) - drop, 0) if n else 0 for n in wl.seq_lens], np.int32)
    return dataclasses.replace(wl, seq_lens=lens)


def _token_call(wl, lens):
    """Append call of the token at position lens[b] - 1 of every sequence with lens[b] > 0."""
    rows_k, rows_v, cu, ctx = [], [], [0], []
    for b in range(wl.batch):
        n = int(lens[b])
        if n > 0:
            r = int(wl.tok_off[b]) + n - 1
            rows_k.append(wl.k_bits[r])
            rows_v.append(wl.v_bits[r])
        cu.append(cu[-1] + (1 if n > 0 else 0))
        ctx.append(max(n - 1, 0))
    Hkv, D = wl.num_kv_heads, wl.head_dim
    k = np.stack(rows_k) if rows_k else np.zeros((0, Hkv, D), np.uint16)
    v = np.stack(rows_v) if rows_v else np.zeros((0, Hkv, D), np.uint16)
    return W.AppendCall(np.ascontiguousarray(k), np.ascontiguousarray(v), np.asarray(cu, np.int32),
                        np.asarray(ctx, np.int32), np.ascontiguousarray(wl.block_table))


@pytest.mark.parametrize("name", ["qwen25_7b_bf16", "qwen3_8b_int8", "long_uint4", "qwen3_8b_fp8"])
def test_full_size_step(name):
    """The benchmark's workloads: the whole pool bit-exact after the fused
    step and every output row within tolerance of the oracle."""
    wl = W.CONFIGS[name]()
    g, o = H.load_both(wl, leave_last=True)
    call = wl.step_call()
    k, v = _rows(wl, call)
    got = _step(g, wl, k, v, wl.seq_lens, 0, early=True)
    assert o.append_call(call) == 0
    H.assert_pools_equal(g, o)
    ref, st = o.decode(wl.q_bits, wl.block_table, wl.seq_lens, wl.softmax_scale)
    assert st == 0
    H.check_attention(got, ref, name)
    assert g.device_error() == (0, 0)
    g.close()


def test_step_refuses_null_token_rows():
    from paged_gqa_decode_02_gb300 import binding as B
    import ctypes
    wl = W.tiny()
    g, _ = H.make_pools(wl)
    L = B.lib()
    st = L.pa_decode_step(g.handle, None, None, None, None, None, 2, 4, 3, 0.125, None, None, 0, 0, None)
    assert st == 1 and b"k_new" in L.pa_last_error()
    assert L.pa_decode_step(g.handle, None, None, None, None, None, 0, 4, 3, 0.125, None, None, 0, 0, None) == 0
    g.close()
