"""Shared helpers for the tests: drive the CUDA library and the CPU oracle on
the same seeded workload and compare them."""
from __future__ import annotations

import numpy as np

from oracle import oracle
from paged_gqa_decode_02_gb300 import workloads as W

BF16_NAN = 0x7FC0
E4M3_NAN = 0x7F
ATOL, RTOL = 2e-3, 1e-2  # decode tolerance: max-abs, and per-row max-abs / max|ref|


def torch_mod():
    import torch
    return torch


def dev(a, dtype=None):
    torch = torch_mod()
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    t = torch.from_numpy(a)
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def host_pool_arrays(gpool):
    """Copy a GPU pool to numpy, in the oracle's naming."""
    v = {k: np.ascontiguousarray(t.contiguous().cpu().numpy()) for k, t in gpool.view().items()}
    out = {}
    if gpool.kv_dtype == "bf16":
        out["k16"] = v["k"].view(np.uint16)
        out["v16"] = v["v"].view(np.uint16)
    else:
        out["kc"], out["vc"] = v["k"], v["v"]
        out["ks"], out["vs"] = v["k_scale"], v["v_scale"]
        if "k_zp" in v:
            out["kz"], out["vz"] = v["k_zp"], v["v_zp"]
    return out


def make_pools(wl, poison=True):
    """An empty GPU pool and an empty oracle pool in the same initial state
    (bf16 and fp8 pools poisoned with NaN so a stray read shows up)."""
    from paged_gqa_decode_02_gb300.binding import PagedKVPool
    g = PagedKVPool(wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim, wl.kv_dtype)
    fill = {"bf16": BF16_NAN, "fp8": E4M3_NAN}.get(wl.kv_dtype, 0) if poison else 0
    o = oracle.OraclePool(wl.kv_dtype, wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim,
                          fill=fill)
    if fill:
        v = g.view()
        v["k"].fill_(fill)
        v["v"].fill_(fill)
    if poison and wl.kv_dtype != "bf16":
        # scales of never-written blocks are NaN on both sides: a read of one
        # (a block the append has not quantised yet) shows up in the output
        v = g.view()
        v["k_scale"].fill_(float("nan"))
        v["v_scale"].fill_(float("nan"))
        o.ks[...] = np.float32(np.nan)
        o.vs[...] = np.float32(np.nan)
    return g, o


def gpu_append(gpool, call, max_new=0):
    torch = torch_mod()
    gpool.append_kv(dev(call.k_bits), dev(call.v_bits), dev(call.cu_new), dev(call.ctx_lens),
                    dev(call.block_table), max_new_per_seq=max_new or call.max_new)


def load_both(wl, leave_last=True):
    """Fill both pools through the append entry point / the oracle append:
    the bulk load, then (with leave_last) the decode step's one-token append."""
    g, o = make_pools(wl)
    calls = wl.fill_calls(leave_last=leave_last)
    if leave_last:
        calls.append(wl.step_call())
    for c in calls:
        gpu_append(g, c)
        assert o.append_call(c) == 0
    return g, o


def assert_pools_equal(gpool, opool):
    h = host_pool_arrays(gpool)
    for name, arr in h.items():
        ref = getattr(opool, name)
        if not np.array_equal(arr.view(np.uint8) if arr.dtype != np.uint8 else arr,
                              ref.view(np.uint8) if ref.dtype != np.uint8 else ref):
            diff = np.argwhere(arr != ref) if arr.dtype != np.float32 else np.argwhere(
                arr.view(np.uint32) != ref.view(np.uint32))
            raise AssertionError(f"pool array {name} differs at {len(diff)} places, first {diff[:5].tolist()}")


def gpu_decode(gpool, wl, num_splits=0, out_fill=float("nan"), path="auto", combine="separate",
               early_plan=False, unit_cost=-1):
    torch = torch_mod()
    gpool.set_decode_path(path, fused_combine=(combine == "fused"), early_plan=early_plan)
    gpool.set_unit_cost(unit_cost)
    out = torch.full((wl.batch, wl.num_q_heads, wl.head_dim), out_fill, dtype=torch.float32,
                     device="cuda")
    gpool.decode(dev(wl.q_bits), dev(wl.block_table), dev(wl.seq_lens), wl.softmax_scale, out=out,
                 num_splits=num_splits)
    torch.cuda.synchronize()
    return out.cpu().numpy().reshape(wl.batch * wl.num_q_heads, wl.head_dim)


def check_attention(got, ref, what=""):
    got = np.asarray(got, np.float64)
    bad_rows = np.where(~np.isfinite(got).all(axis=1))[0]
    assert bad_rows.size == 0, f"{what}: non-finite outputs in rows {bad_rows[:16].tolist()} of {got.shape[0]}"
    err = np.abs(got - ref)
    max_abs = float(err.max()) if err.size else 0.0
    row_rel = err.max(axis=1) / np.maximum(np.abs(ref).max(axis=1), 1e-6) if err.size else np.zeros(1)
    assert max_abs <= ATOL, f"{what}: max-abs error {max_abs:.3g} > {ATOL}"
    assert float(row_rel.max()) <= RTOL, f"{what}: max row-relative error {row_rel.max():.3g} > {RTOL}"
    return max_abs, float(row_rel.max())


def sample_rows(wl, n=48, seed=0):
    """Rows (b*Hq + h) to check at full size: longest, shortest, first, last
    and random ones."""
    rng = np.random.default_rng(seed)
    Hq = wl.num_q_heads
    bs = [int(np.argmax(wl.seq_lens)), int(np.argmin(wl.seq_lens)), 0, wl.batch - 1]
    rows = [b * Hq + h for b in bs for h in (0, Hq - 1)]
    rows += list(rng.integers(0, wl.batch * Hq, size=max(0, n - len(rows))))
    return np.unique(np.asarray(rows, np.int64))
