"""Block tables from the host block manager drive the append and decode
entry points. Sequences share prefix-cached blocks, a forked sequence gets a
copy-on-write page copy (pa_copy_blocks), and both the pool and the attention
match the oracle fed the same tables and copies."""
import numpy as np
import pytest

from oracle import oracle
from paged_gqa_decode_02_gb300 import binding as B
from paged_gqa_decode_02_gb300 import workloads as W
from tests import harness as H

pytestmark = pytest.mark.gpu


def _kv_for(tokens, Hkv, D):
    """K/V of every position as a function of the token prefix up to it, so that
    sequences with the same prefix have the same KV there."""
    k = np.empty((len(tokens), Hkv, D), np.uint16)
    v = np.empty_like(k)
    h = 17
    for t, tok in enumerate(tokens):
        h = (h * 1000003 + int(tok) + 1) % (1 << 61)
        r = np.random.default_rng([h % (1 << 32), h >> 32])
        k[t] = W.f32_to_bf16_bits(r.standard_normal((Hkv, D)).astype(np.float32))
        v[t] = W.f32_to_bf16_bits(r.standard_normal((Hkv, D)).astype(np.float32))
    return k, v


def _copy_oracle_block(o, src, dst):
    for name in ("k16", "v16", "kc", "vc", "ks", "vs", "kz", "vz"):
        a = getattr(o, name)
        if a is not None:
            a[dst] = a[src]


@pytest.mark.parametrize("dt", ["bf16", "uint8", "uint4", "fp8"])
def test_block_manager_tables_drive_append_and_decode(dt):
    bs, Hkv, Hq, D, nb, MB = 16, 2, 8, 128, 48, 8
    rng = np.random.default_rng(11)
    bm = B.BlockManager(nb, bs)
    g, o = H.make_pools(W.make_case("bm", 11, 1, Hq, Hkv, D, bs, dt, [1], extra_blocks=nb - 1))
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
        return cached

    def step(sid, tok):
        copies = bm.append_tokens(sid, [tok])
        for src, dst in copies:
            g.copy_blocks([src], [dst])
            _copy_oracle_block(o, src, dst)
        table, _ = bm.block_table(sid, MB)
        full = toks[sid] + [tok]
        k, v = _kv_for(full, Hkv, D)
        n0 = len(toks[sid])
        args = (k[n0:], v[n0:], np.array([0, 1], np.int32), np.array([n0], np.int32), table[None, :])
        g.append_kv(*(H.dev(a) for a in args), max_new_per_seq=1)
        assert o.append(*args) == 0
        toks[sid] = full
        return copies

    base = [int(x) for x in rng.integers(0, 50, 40)]  # 2 full blocks + 8 tokens
    assert admit(1, base) == 0
    assert admit(2, base[:32] + [1, 2, 3]) == 32  # shares sequence 1's full blocks
    assert admit(3, [int(x) for x in rng.integers(50, 99, 20)]) == 0
    bm.fork(1, 4)
    toks[4] = list(toks[1])
    assert len(step(4, 77)) == 1  # the shared partial tail is copied first
    assert step(1, 78) == []  # sequence 1's tail is private again
    assert step(2, 79) == []

    H.assert_pools_equal(g, o)
    sids = [1, 2, 3, 4]
    table = np.stack([bm.block_table(s, MB)[0] for s in sids]).astype(np.int32)
    lens = np.array([len(toks[s]) for s in sids], np.int32)
    q = W.f32_to_bf16_bits(rng.standard_normal((len(sids), Hq, D)).astype(np.float32))
    scale = 1.0 / np.sqrt(D)
    ref, st = o.decode(q, table, lens, scale)
    assert st == 0
    out = g.decode(H.dev(q), H.dev(table), H.dev(lens), scale)
    H.check_attention(out.cpu().numpy().reshape(-1, D), ref, f"block-manager tables {dt}")
    assert g.device_error() == (0, 0)
    g.close()


def test_decode_step_replays_from_a_cuda_graph():
    """One decode step (append the step's token, decode, combine) captured in a
    CUDA graph and replayed gives the same outputs as direct calls. The step
    is idempotent for a bf16 pool (the append copies the same token again)."""
    torch = H.torch_mod()
    wl = W.make_case("graph", 12, 6, 28, 4, 128, 16, "bf16", [700, 33, 1500, 1, 257, 4096], extra_blocks=2)
    g, _ = H.load_both(wl, leave_last=False)
    g.set_decode_path("auto", early_plan=True)
    sc = wl.step_call()
    k, v, cu, ctx = H.dev(sc.k_bits), H.dev(sc.v_bits), H.dev(sc.cu_new), H.dev(sc.ctx_lens)
    table, lens, q = H.dev(wl.block_table), H.dev(wl.seq_lens), H.dev(wl.q_bits)
    out = torch.empty((wl.batch, wl.num_q_heads, wl.head_dim), dtype=torch.float32, device="cuda")
    ws = g.workspace(wl.batch, wl.num_q_heads)

    def step():
        g.append_kv(k, v, cu, ctx, table, max_new_per_seq=1)
        g.decode(q, table, lens, wl.softmax_scale, out=out, workspace=ws)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(2):  # first calls set the kernels' attributes, outside the capture
            step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    ref = out.clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step()
    for _ in range(3):
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
    assert g.device_error() == (0, 0)
    g.close()


def test_fused_combine_replays_from_a_cuda_graph_with_new_queries():
    """The in-kernel merge (PA_DECODE_FUSED_COMBINE) captured in a CUDA graph:
    every replay keeps the captured call's ticket tag, so the merging slice
    must leave its tickets cleared. New queries are copied into the captured
    buffer before each replay and every replay must match the oracle for them
    (a stale ticket would leave split rows unmerged, holding the last replay's
    values)."""
    torch = H.torch_mod()
    wl = W.make_case("graph_fused", 13, 6, 28, 4, 128, 16, "bf16", [700, 33, 1500, 1, 257, 4096], extra_blocks=2)
    g, o = H.load_both(wl, leave_last=False)
    g.set_decode_path("auto", fused_combine=True, early_plan=False)
    table, lens = H.dev(wl.block_table), H.dev(wl.seq_lens)
    q = H.dev(wl.q_bits)
    out = torch.empty((wl.batch, wl.num_q_heads, wl.head_dim), dtype=torch.float32, device="cuda")
    ws = g.workspace(wl.batch, wl.num_q_heads)

    def call():
        g.decode(q, table, lens, wl.softmax_scale, out=out, workspace=ws)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(2):
            call()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        call()
    rng = np.random.default_rng(77)
    for r in range(3):
        qb = W.f32_to_bf16_bits(rng.standard_normal(wl.q_bits.shape, dtype=np.float32))
        q.copy_(H.dev(qb))
        out.fill_(float("nan"))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        ref, st = o.decode(qb, wl.block_table, wl.seq_lens, wl.softmax_scale)
        assert st == 0
        H.check_attention(out.cpu().numpy().reshape(-1, wl.head_dim), ref, f"fused graph replay {r}")
    assert g.device_error() == (0, 0)
    g.close()
