"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs. Quantised append must match bit-exactly (codes, scales,
zero points); decode within max-abs 2e-3 and per-row relative 1e-2."""
import numpy as np
import pytest

from paged_gqa_decode_02_gb300 import workloads as W
from tests import harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_gqa_decode_02_gb300 import build
    build.build()


def _paths(dt, head_dim=128):
    """Decode kernels that serve a pool: tensor cores for bf16, and for
    quantised pools with head_dim 128; the CUDA-core kernel everywhere."""
    if dt == "bf16" or head_dim == 128:
        return ["cuda_core", "tensor_core"]
    return ["cuda_core"]


@pytest.mark.parametrize("combine", ["fused", "separate"])
@pytest.mark.parametrize("path", ["cuda_core", "tensor_core"])
@pytest.mark.parametrize("splits", [0, 1, 2, 3, 1000])
def test_tiny_config(splits, path, combine):
    wl = W.tiny()
    g, o = H.load_both(wl)
    H.assert_pools_equal(g, o)
    ref, st = o.decode(wl.q_bits, wl.block_table, wl.seq_lens, wl.softmax_scale)
    assert st == 0
    got = H.gpu_decode(g, wl, num_splits=splits, path=path, combine=combine)
    H.check_attention(got, ref, f"tiny splits={splits} {path} {combine}")
    assert g.device_error() == (0, 0)


@pytest.mark.parametrize("dt", ["bf16", "uint8", "uint4", "fp8"])
@pytest.mark.parametrize("seed", range(8))
def test_random_small(seed, dt):
    wl = W.random_small(seed, dt)
    g, o = H.load_both(wl)
    H.assert_pools_equal(g, o)
    ref, st = o.decode(wl.q_bits, wl.block_table, wl.seq_lens, wl.softmax_scale)
    assert st == 0
    for path in _paths(dt, wl.head_dim):
        for splits in (0, 1, 5, 10 ** 4):
            for combine in ("fused", "separate"):
                got = H.gpu_decode(g, wl, num_splits=splits, path=path, combine=combine,
                                   early_plan=(splits % 2 == 1))
                H.check_attention(got, ref, f"{wl.name} {dt} splits={splits} {path} {combine}")
    assert g.device_error() == (0, 0)


@pytest.mark.parametrize("dt", ["bf16", "uint8", "uint4", "fp8"])
@pytest.mark.parametrize("block_size", [16, 32])
def test_unit_cost_partition(block_size, dt):
    """The cost-balanced partition moves pages between thread blocks but never
    changes the result: phantom pages per unit from none to far more than a
    unit's pages (slices that hold only phantom positions, units cut into
    many slices), empty and one-token sequences, with the separate and the
    in-kernel merge."""
    seq = [0, 1, 17, 200, 33, 0, 512, 3, 90]
    wl = W.make_case(f"unit_cost_bs{block_size}", 93, len(seq), 8, 2, 128, block_size, dt, seq, extra_blocks=2,
                     channel_offset_sigma=0.5 if dt != "bf16" else None)
    g, o = H.load_both(wl)
    ref, st = o.decode(wl.q_bits, wl.block_table, wl.seq_lens, wl.softmax_scale)
    assert st == 0
    for path in _paths(dt, wl.head_dim):
        for unit_cost in (0, 1, 5, 40, 4096):
            for splits, combine, early in ((0, "separate", True), (7, "fused", False), (300, "separate", False)):
                got = H.gpu_decode(g, wl, num_splits=splits, path=path, combine=combine, early_plan=early,
                                   unit_cost=unit_cost)
                H.check_attention(got, ref, f"{wl.name} {dt} unit_cost={unit_cost} splits={splits} {path} {combine}")
    assert g.device_error() == (0, 0)
    with pytest.raises(Exception):
        g.set_unit_cost(5000)


@pytest.mark.parametrize("dt", ["bf16", "uint8", "uint4", "fp8"])
def test_multi_step_tail_requant(dt):
    """Several decode steps, each appending one token per sequence into a
    partly filled block (re-quantised), then attending."""
    wl = W.make_case("steps", 31, 3, 8, 2, 128, 16, dt, [20, 33, 7], extra_blocks=3,
                     channel_offset_sigma=0.5 if dt != "bf16" else None)
    g, o = H.make_pools(wl)
    first = wl.fill_calls(leave_last=True)[0]
    H.gpu_append(g, first)
    assert o.append_call(first) == 0
    step = wl.step_call()
    for _ in range(3):
        H.gpu_append(g, step)
        assert o.append_call(step) == 0
        H.assert_pools_equal(g, o)
        ref, _ = o.decode(wl.q_bits, wl.block_table, wl.seq_lens, wl.softmax_scale)
        for path in _paths(dt, wl.head_dim):
            H.check_attention(H.gpu_decode(g, wl, path=path), ref, f"steps {dt} {path}")


def test_empty_and_single_token_sequences():
    wl = W.make_case("edge", 41, 5, 12, 4, 64, 16, "bf16", [0, 1, 16, 0, 17], extra_blocks=2)
    g, o = H.load_both(wl, leave_last=False)
    ref, _ = o.decode(wl.q_bits, wl.block_table, wl.seq_lens, wl.softmax_scale)
    for path in _paths("bf16"):
        for splits in (0, 1, 7):
            for combine in ("fused", "separate"):
                got = H.gpu_decode(g, wl, num_splits=splits, path=path, combine=combine)
                H.check_attention(got, ref, f"edge splits={splits} {path} {combine}")
                assert np.all(got.reshape(5, 12, 64)[[0, 3]] == 0)


def test_bad_table_entry_sets_error_word_and_gpu_stays_usable():
    from paged_gqa_decode_02_gb300 import binding as B
    wl = W.random_small(3, "uint8")
    g, o = H.load_both(wl)
    bad = wl.block_table.copy()
    bad[0, 0] = wl.num_blocks + 5
    torch = H.torch_mod()
    out = torch.zeros((wl.batch, wl.num_q_heads, wl.head_dim), dtype=torch.float32, device="cuda")
    g.decode(H.dev(wl.q_bits), H.dev(bad), H.dev(wl.seq_lens), wl.softmax_scale, out=out)
    st, flags = g.device_error()
    assert st == 5 and flags & B.DEVERR_BLOCK_TABLE
    bad_len = wl.seq_lens.copy()
    bad_len[-1] = wl.max_blocks * wl.block_size + 1
    g.decode(H.dev(wl.q_bits), H.dev(wl.block_table), H.dev(bad_len), wl.softmax_scale, out=out)
    st, flags = g.device_error()
    assert st == 5 and flags & B.DEVERR_SEQ_LEN
    # a clean call afterwards is still correct
    ref, _ = o.decode(wl.q_bits, wl.block_table, wl.seq_lens, wl.softmax_scale)
    H.check_attention(H.gpu_decode(g, wl), ref, "after error")
    assert g.device_error() == (0, 0)


def test_host_validation_errors():
    from paged_gqa_decode_02_gb300 import binding as B
    wl = W.tiny()
    g, _ = H.make_pools(wl)
    torch = H.torch_mod()
    q = H.dev(wl.q_bits)
    with pytest.raises(B.PagedAttnError) as e:
        g.decode(q[:, :3], H.dev(wl.block_table), H.dev(wl.seq_lens), 0.125)  # 3 heads, Hkv = 2
    assert e.value.status == 1
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(B.PagedAttnError) as e:
        g.decode(q, H.dev(wl.block_table), H.dev(wl.seq_lens), 0.125, workspace=ws)
    assert e.value.status == 3
    # out must be 16-byte aligned (rows are written as float4)
    n = wl.batch * wl.num_q_heads * wl.head_dim
    out_off = torch.empty(n + 1, dtype=torch.float32, device="cuda")[1:].view(wl.batch, wl.num_q_heads, wl.head_dim)
    with pytest.raises(B.PagedAttnError) as e:
        g.decode(q, H.dev(wl.block_table), H.dev(wl.seq_lens), 0.125, out=out_off)
    assert e.value.status == 1 and "16-byte" in str(e.value)


FULL = ["qwen25_7b_bf16", "qwen3_8b_int8", "long_uint4", "prefix_mix", "qwen3_8b_fp8"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_config(name):
    """Full-size workloads: the whole pool bit-exact after the bulk append and
    the decode step's append; attention on every output row (the oracle,
    OpenMP over the host's cores, computes them all), in the automatic
    launch configuration the benchmark times and with one forced split count."""
    wl = W.CONFIGS[name]()
    g, o = H.load_both(wl)
    H.assert_pools_equal(g, o)
    ref, st = o.decode(wl.q_bits, wl.block_table, wl.seq_lens, wl.softmax_scale)
    assert st == 0
    for path in _paths(wl.kv_dtype, wl.head_dim):
        for splits, combine, early in ((0, "fused", False), (97, "fused", True), (0, "separate", True),
                                       (0, "separate", False)):
            got = H.gpu_decode(g, wl, num_splits=splits, path=path, combine=combine, early_plan=early)
            H.check_attention(got, ref, f"{name} splits={splits} {path} {combine} early={early}")
    assert g.device_error() == (0, 0)


@pytest.mark.parametrize("dt", ["bf16", "uint8", "fp8"])
def test_slices_longer_than_a_window(dt):
    """One or two slices over thousands of pages: a thread block walks its
    slice in several windows and runs continue across window boundaries."""
    wl = W.make_case("long_slices", 55, 3, 8, 2, 64, 16, dt, [21000, 5, 9000], extra_blocks=1,
                     channel_offset_sigma=0.5 if dt != "bf16" else None)
    g, o = H.load_both(wl)
    H.assert_pools_equal(g, o)
    ref, st = o.decode(wl.q_bits, wl.block_table, wl.seq_lens, wl.softmax_scale)
    assert st == 0
    for path in _paths(dt, wl.head_dim):
        for splits in (1, 2, 3):
            got = H.gpu_decode(g, wl, num_splits=splits, path=path)
            H.check_attention(got, ref, f"long slices {dt} splits={splits} {path}")
    assert g.device_error() == (0, 0)


@pytest.mark.parametrize("early_plan", [False, True])
@pytest.mark.parametrize("combine", ["fused", "separate"])
@pytest.mark.parametrize("splits", [0, 300, 2000])
def test_many_slices_per_sequence(splits, combine, early_plan):
    """Units cut into many slices (up to 32, and past the combine's 64-slice
    rounds) with a 7-head group; with early_plan the combine works out each
    unit's slices from the lengths before waiting on the decode kernel."""
    wl = W.make_case("many_slices", 92, 3, 28, 4, 128, 16, "bf16", [700, 33, 1500], extra_blocks=2)
    g, o = H.load_both(wl)
    ref, st = o.decode(wl.q_bits, wl.block_table, wl.seq_lens, wl.softmax_scale)
    assert st == 0
    for path in _paths("bf16"):
        got = H.gpu_decode(g, wl, num_splits=splits, path=path, combine=combine, early_plan=early_plan)
        H.check_attention(got, ref, f"many slices splits={splits} {path} {combine} early={early_plan}")
    assert g.device_error() == (0, 0)


@pytest.mark.parametrize("dt", ["bf16", "uint8", "uint4", "fp8"])
def test_decode_writes_nothing_outside_out_and_workspace(dt):
    """Canaries: guard regions before and after the output and the workspace
    keep their bytes through decodes with many slices, both merge modes and
    the early plan (a stray write past a slot or row would change them)."""
    torch = H.torch_mod()
    seq = [300, 1, 0, 45, 1000, 17, 2]
    wl = W.make_case(f"canary_{dt}", 77, len(seq), 8, 2, 128, 16, dt, seq, extra_blocks=1,
                     channel_offset_sigma=None if dt == "bf16" else 0.5)
    g, o = H.load_both(wl)
    ref, st = o.decode(wl.q_bits, wl.block_table, wl.seq_lens, wl.softmax_scale)
    assert st == 0
    B, Hq, D = wl.batch, wl.num_q_heads, wl.head_dim
    GW, GO = 4096, 1024  # guard bytes around the workspace, guard floats around out
    q, table, lens = H.dev(wl.q_bits), H.dev(wl.block_table), H.dev(wl.seq_lens)
    for splits, combine, early in ((0, "separate", True), (7, "fused", False), (300, "separate", False),
                                   (1000, "fused", True)):
        g.set_decode_path("auto", fused_combine=(combine == "fused"), early_plan=early)
        n = g.workspace_bytes(B, Hq, splits)
        wbuf = torch.full((n + 2 * GW,), 0xA5, dtype=torch.uint8, device="cuda")
        ws = wbuf[GW:GW + n]
        ws.zero_()
        obuf = torch.full((B * Hq * D + 2 * GO,), 12345.0, dtype=torch.float32, device="cuda")
        out = obuf[GO:GO + B * Hq * D].view(B, Hq, D)
        out.fill_(float("nan"))
        g.decode(q, table, lens, wl.softmax_scale, out=out, workspace=ws, num_splits=splits)
        torch.cuda.synchronize()
        what = f"canary {dt} splits={splits} {combine} early={early}"
        assert bool((wbuf[:GW] == 0xA5).all()) and bool((wbuf[GW + n:] == 0xA5).all()), what + ": workspace guard"
        assert bool((obuf[:GO] == 12345.0).all()) and bool((obuf[GO + B * Hq * D:] == 12345.0).all()), what + ": out guard"
        H.check_attention(out.cpu().numpy().reshape(-1, D), ref, what)
    assert g.device_error() == (0, 0)
    g.close()


@pytest.mark.parametrize("dt", ["bf16", "uint8"])
def test_batch_beyond_the_plan_caches(dt):
    """More sequences than the decode kernel has threads (the plan's multi-pass
    scan) and than it keeps lengths of in shared memory (later lengths are
    read again from global memory), with empty and one-token sequences mixed
    in."""
    rng = np.random.default_rng([57, 0])
    seq = rng.integers(0, 40, 5000).astype(np.int32)
    wl = W.make_case(f"big_batch_{dt}", 57, seq.size, 4, 1, 64, 16, dt, seq,
                     channel_offset_sigma=None if dt == "bf16" else 0.5)
    g, o = H.load_both(wl)
    rows = H.sample_rows(wl, n=256)
    ref, st = o.decode(wl.q_bits, wl.block_table, wl.seq_lens, wl.softmax_scale, rows=rows)
    assert st == 0
    for splits, combine, early in ((0, "separate", True), (97, "fused", False), (3000, "separate", False)):
        got = H.gpu_decode(g, wl, num_splits=splits, combine=combine, early_plan=early)
        assert np.isfinite(got).all()
        H.check_attention(got[rows], ref, f"big batch {dt} splits={splits} {combine}")
        empty = np.flatnonzero(wl.seq_lens == 0)
        assert np.all(got.reshape(wl.batch, -1)[empty] == 0)
    assert g.device_error() == (0, 0)
    g.close()
