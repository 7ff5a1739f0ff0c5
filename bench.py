"""Benchmark: one decode step of paged GQA attention per step -- append the
step's new token of every sequence (kv_quant_append), then attend
(paged_gqa_decode + split-KV combine) -- on the Qwen2.5-7B-shaped workload
(batch 32, 28 Q / 4 KV heads, head_dim 128, block 16, seq_lens U[512, 4096],
bf16 KV), synthetic seeded data.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--splits S]

Prints one JSON line. value = decode tokens per second (batch / step time),
whole job over all ranks. The L2 cache is flushed (a 256 MiB write) between
timed steps, outside the per-step CUDA-event brackets. Under torchrun every
rank runs its own replica of the workload (the path needs no exchange between
GPUs): weak scaling.
"""
from __future__ import annotations

import argparse
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged GQA decode attention: tokens/s and achieved HBM GB/s (% of GB300 peak)"
WORKLOAD_TEXT = {
    "qwen25_7b_bf16": "Qwen2.5-7B-shaped decode: batch 32, 28 Q / 4 KV heads, head_dim 128, block 16, "
                      "seq_lens U[512,4096], bf16 KV",
    "qwen3_8b_int8": "Qwen3-8B-shaped uint8 KV: batch 64, 32 Q / 8 KV heads, head_dim 128, block 16, "
                     "seq_lens U[1,8192]",
    "long_uint4": "long-context uint4 KV: batch 4, 32 Q / 8 KV heads, head_dim 128, block 32, 32768 tokens each",
    "qwen3_8b_fp8": "Qwen3-8B-shaped fp8 (E4M3) KV: batch 64, 32 Q / 8 KV heads, head_dim 128, block 16, "
                    "seq_lens U[1,8192]",
    "prefix_mix": "continuous-batching mix with prefix cache: batch 256, 28 Q / 4 KV heads, head_dim 128, "
                  "block 16, lognormal(median 1000) lengths, 8x32 sequences share 512-token prefixes, bf16 KV",
    "tiny": "tiny: batch 2, 4 Q / 2 KV heads, head_dim 64, block 16, seq_lens {37,5}, bf16 KV",
}


PROFILE_FOR = {"qwen25_7b_bf16": "profiles/paged_gqa_decode_qwen25_7b_bf16.md",
               "qwen3_8b_int8": "profiles/paged_gqa_decode_qwen3_8b_int8.md",
               "long_uint4": "profiles/paged_gqa_decode_long_uint4.md"}


# The consumer sections of the decode source each workload's tensor-core
# kernel compiles from; the other consumers' sections do not reach its code.
_CONSUMER_SECTIONS = ("consumer math (CUDA cores)", "consumer math (tensor cores)",
                      "consumer math (tensor cores, uint8 KV)", "consumer math (tensor cores, uint4 KV)",
                      "consumer math (tensor cores, fp8 KV)")
_USES = {"qwen25_7b_bf16": "consumer math (tensor cores)", "prefix_mix": "consumer math (tensor cores)",
         "qwen3_8b_int8": "consumer math (tensor cores, uint8 KV)",
         "long_uint4": "consumer math (tensor cores, uint4 KV)",
         "qwen3_8b_fp8": "consumer math (tensor cores, fp8 KV)"}


_C_TOKENS = re.compile(r'"(?:\\.|[^"\\\n])*"|\'(?:\\.|[^\'\\\n])*\'|//[^\n]*|/\*.*?\*/', re.S)


def _code_only(text):
    """C/CUDA source with its comments removed, trailing blanks stripped and
    empty lines dropped: two sources that differ only in comments or blank
    lines compile to the same kernel and give the same text."""
    text = _C_TOKENS.sub(lambda m: " " if m.group(0)[0] == "/" else m.group(0), text)
    return "\n".join(l.rstrip() for l in text.splitlines() if l.strip())


def kernel_source_hash(workload, decode_src=None, common_src=None):
    """sha256 (16 hex digits) of the code this workload's tensor-core decode
    kernel is compiled from: the decode-kernel and common sources without the
    sections of the consumers it does not use, comments and blank lines
    removed. The sources default to the files in the tree."""
    import hashlib
    csrc = os.path.join(ROOT, "paged_gqa_decode_02_gb300", "csrc")
    src = decode_src if decode_src is not None else open(os.path.join(csrc, "pa_decode_kernels.cuh")).read()
    common = common_src if common_src is not None else open(os.path.join(csrc, "pa_common.cuh")).read()
    keep = _USES[workload]
    parts = src.split("// " + "-" * 66 + " ")
    kept = [parts[0]] + [x for x in parts[1:] if not (x.split("\n", 1)[0].strip() in _CONSUMER_SECTIONS
                                                       and x.split("\n", 1)[0].strip() != keep)]
    return hashlib.sha256((_code_only("".join(kept)) + "\n" + _code_only(common)).encode()).hexdigest()[:16]


def _traffic(workload, path):
    """DRAM bytes per decode launch from the committed ncu summary, or None
    when there is none for this workload or the kernel's source changed since."""
    rel = PROFILE_FOR.get(workload)
    if rel is None or path not in ("auto", "tensor_core"):
        return None
    try:
        text = open(os.path.join(ROOT, rel)).read()
        fields = dict(l.split(": ", 1) for l in text.splitlines() if l.startswith(("traffic_", "kernel_source_")))
        if kernel_source_hash(workload) != fields["kernel_source_sha256_16"].strip():
            return None
        return int(fields["traffic_bytes_per_launch"])
    except Exception:
        return None


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9], parts[4]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[2]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group("gloo")
        return dist, int(os.environ.get("RANK", "0")), ws
    return None, 0, 1


def _max_over_ranks(dist, x):
    if dist is None:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _barrier(dist):
    if dist is not None:
        dist.barrier()


def run_ours(args):
    import torch
    from paged_gqa_decode_02_gb300 import build as pbuild
    from paged_gqa_decode_02_gb300 import workloads as W
    from paged_gqa_decode_02_gb300.binding import PagedKVPool
    from paged_gqa_decode_02_gb300.metrics import decode_bytes

    dist, rank, world = _dist()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if rank == 0:
        pbuild.build()
    _barrier(dist)
    wl = W.CONFIGS[args.workload]()
    dev = torch.device("cuda", local)
    pool = PagedKVPool(wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim, wl.kv_dtype, local)
    pool.set_decode_path(args.path, fused_combine=(args.combine == "fused"),
                         early_plan=not args.no_early_plan)
    pool.set_unit_cost(args.unit_cost)

    def d(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        return torch.from_numpy(a).to(dev)

    # several query tokens per sequence (chunked prefill / speculative
    # verification): the step appends the last n_q tokens and attends with all
    n_q = args.query_tokens
    for c in wl.fill_calls(leave_last=(n_q == 1)):
        pool.append_kv(d(c.k_bits), d(c.v_bits), d(c.cu_new), d(c.ctx_lens), d(c.block_table),
                       max_new_per_seq=c.max_new)
    step = wl.step_call(n_q)
    st_k, st_v, st_cu, st_ctx = d(step.k_bits), d(step.v_bits), d(step.cu_new), d(step.ctx_lens)
    B, Hq, D = wl.batch, wl.num_q_heads, wl.head_dim
    q_bits = wl.q_bits if n_q == 1 else W.multi_token_queries(100, B, n_q, Hq, D)
    table, seq_lens, q = d(wl.block_table), d(wl.seq_lens), d(q_bits)
    out = torch.empty(q_bits.shape, dtype=torch.float32, device=dev)
    ws = pool.workspace(B, Hq, args.splits)
    splits_used = pool.num_splits(args.splits)

    def decode_call(q_, table_, lens_):
        if n_q == 1:
            pool.decode(q_, table_, lens_, wl.softmax_scale, out=out, workspace=ws, num_splits=args.splits)
        else:
            pool.decode_multi(q_, table_, lens_, wl.softmax_scale, out=out, num_splits=args.splits)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def one_step():
        # append then decode back to back, as a decode loop runs them (the
        # decode's planning may overlap the append; see --no-early-plan)
        pool.append_kv(st_k, st_v, st_cu, st_ctx, table, max_new_per_seq=n_q)
        decode_call(q, table, seq_lens)

    for _ in range(max(3, args.warmup)):
        flush.fill_(1)
        one_step()
    torch.cuda.synchronize()
    st, flags = pool.device_error()
    assert st == 0 and flags == 0, f"device error word {flags:#x} during warm-up"

    clocks = ClockSampler(local)
    clocks.start()
    # soak so that the clock record covers a loaded GPU before and during timing
    t_end = time.time() + 1.0
    while time.time() < t_end:
        flush.fill_(1)
        one_step()
    torch.cuda.synchronize()

    K = args.steps
    e0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    e2 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    _barrier(dist)
    torch.cuda.synchronize()
    for i in range(K):
        flush.fill_(1)
        e0[i].record(stream)
        one_step()
        e2[i].record(stream)
    torch.cuda.synchronize()
    _barrier(dist)
    # roofline of the decode call alone: a second pass of K calls, each
    # bracketed by events (L2 flushed before each)
    d0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    d1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for i in range(K):
        flush.fill_(1)
        d0[i].record(stream)
        decode_call(q, table, seq_lens)
        d1[i].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    step_ms = [e0[i].elapsed_time(e2[i]) for i in range(K)]
    dec_ms = [d0[i].elapsed_time(d1[i]) for i in range(K)]
    st, flags = pool.device_error()
    assert st == 0 and flags == 0, f"device error word {flags:#x} during timing"
    t_step = statistics.mean(step_ms) / 1e3
    t_dec = statistics.mean(dec_ms) / 1e3
    t_step_max = _max_over_ranks(dist, t_step)
    t_dec_max = _max_over_ranks(dist, t_dec)

    # ---- e2e through the public API with host buffers (pinned), copies inside the region
    h_in = {k: torch.from_numpy(np.ascontiguousarray(v).view(np.int16) if v.dtype == np.uint16 else
                                np.ascontiguousarray(v)).pin_memory()
            for k, v in (("k", step.k_bits), ("v", step.v_bits), ("cu", step.cu_new), ("ctx", step.ctx_lens),
                         ("table", wl.block_table), ("lens", wl.seq_lens), ("q", q_bits))}
    h_out = torch.empty(q_bits.shape, dtype=torch.float32).pin_memory()
    d_in = {k: torch.empty_like(v, device=dev) for k, v in h_in.items()}
    bi = sum(v.numel() * v.element_size() for v in h_in.values())
    bo = h_out.numel() * h_out.element_size()
    Ke = max(10, min(K, 200))
    e2e_ms = []
    for i in range(Ke + 3):
        flush.fill_(1)
        a = torch.cuda.Event(enable_timing=True)
        z = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for k in d_in:
            d_in[k].copy_(h_in[k], non_blocking=True)
        pool.append_kv(d_in["k"], d_in["v"], d_in["cu"], d_in["ctx"], d_in["table"], max_new_per_seq=n_q)
        decode_call(d_in["q"], d_in["table"], d_in["lens"])
        h_out.copy_(out, non_blocking=True)
        z.record(stream)
        z.synchronize()
        if i >= 3:
            e2e_ms.append(a.elapsed_time(z))
    t_e2e = _max_over_ranks(dist, statistics.mean(e2e_ms) / 1e3)

    nb = decode_bytes(wl, n_q)
    peak, peak_kind = _peaks()
    achieved = nb["algorithmic"] / t_dec_max / 1e9
    res = {
        "metric": METRIC,
        "value": world * B * n_q / t_step_max,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": t_step_max * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if wl.kv_dtype == "bf16" else f"{wl.kv_dtype} codes, fp32 math",
        "data": "synthetic (seeded N(0,1) bf16 q/K/V, block tables from a seeded permutation)",
        "config": {"workload": WORKLOAD_TEXT[args.workload], "name": args.workload, "batch": B,
                   "num_q_heads": Hq, "num_kv_heads": wl.num_kv_heads, "head_dim": D,
                   "block_size": wl.block_size, "kv_dtype": wl.kv_dtype,
                   "tokens_cached": nb["tokens_scanned"], "num_splits": splits_used,
                   "step": (f"append {n_q} token(s)/seq (kv_quant_append) + paged_gqa_decode"
                            + (f" with {n_q} causal query tokens per sequence" if n_q > 1 else "")
                            + " (split-KV merge: " + (args.combine if n_q == 1 else "separate") + ")"),
                   "query_tokens": n_q,
                   "decode_path": args.path,
                   "early_plan": not args.no_early_plan,
                   "unit_cost": args.unit_cost,
                   "l2": "flushed before every timed step (256 MiB write, outside the event brackets)",
                   "parallelism": f"replicas x{world} (no exchange)"},
        "hbm_gbs": achieved,
        "decode_us": t_dec_max * 1e6,
        "median_us": {"step": statistics.median(step_ms) * 1e3, "decode": statistics.median(dec_ms) * 1e3},
        "kv_tokens_per_s": world * nb["tokens_scanned"] / t_dec_max,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": _traffic(args.workload, args.path) if n_q == 1 else None,
                     "peak_kind": f"{peak_kind} (copy bandwidth, MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "algorithmic_bytes_per_launch": nb["algorithmic"],
                     "timed": "pa_decode call (decode kernel + split-KV combine) alone, CUDA events on the "
                              "launch stream, a second pass of K calls after the K timed steps"},
        "e2e": {"value": world * B * n_q / t_e2e, "unit": "tokens/s", "h2d_bytes_per_step": bi,
                "d2h_bytes_per_step": bo},
        "gpu_launches": 3 * K,
        "clocks": clk,
    }
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(wl, args.cpu_seqs, n_q)
    if rank == 0:
        print(json.dumps(res), flush=True)
    pool.close()


def _oracle_setup(wl, n_seq, n_q=1):
    """Oracle pool holding the first n_seq sequences' caches (setup, untimed)."""
    from oracle import oracle
    o = oracle.OraclePool(wl.kv_dtype, wl.num_blocks, wl.num_kv_heads, wl.block_size, wl.head_dim)
    for c in wl.fill_calls(leave_last=(n_q == 1)):
        o.append_call(c)
    step = wl.step_call(n_q)
    keep = np.arange(n_seq)
    per = n_q * wl.num_q_heads  # output rows per sequence
    rows = np.concatenate([np.arange(b * per, (b + 1) * per) for b in keep]).astype(np.int64)
    cu = np.concatenate([[0], np.cumsum(np.diff(step.cu_new)[keep])]).astype(np.int32)
    sel = np.concatenate([np.arange(step.cu_new[b], step.cu_new[b + 1]) for b in keep]).astype(np.int64)
    sub = (step.k_bits[sel], step.v_bits[sel], cu, step.ctx_lens[keep], step.block_table[keep])
    return o, sub, rows


def _oracle_step(wl, o, sub, rows, n_q=1, q_multi=None):
    st = o.append(*sub)
    if n_q == 1:
        out, st2 = o.decode(wl.q_bits, wl.block_table, wl.seq_lens, wl.softmax_scale, rows=rows)
    else:
        out, st2 = o.decode_multi(q_multi, wl.block_table, wl.seq_lens, wl.softmax_scale, rows=rows)
    assert st == 0 and st2 == 0
    return out


def cpu_baseline(wl, n_seq, n_q=1):
    from oracle import oracle
    from paged_gqa_decode_02_gb300 import workloads as W
    n_seq = min(n_seq, wl.batch)
    o, sub, rows = _oracle_setup(wl, n_seq, n_q)
    qm = None if n_q == 1 else W.multi_token_queries(100, wl.batch, n_q, wl.num_q_heads, wl.head_dim)
    _oracle_step(wl, o, sub, rows, n_q, qm)
    reps, t0 = 0, time.perf_counter()
    while True:
        _oracle_step(wl, o, sub, rows, n_q, qm)
        reps += 1
        if time.perf_counter() - t0 > 10.0 or reps >= 20:
            break
    t = (time.perf_counter() - t0) / reps
    return {"value": n_seq * n_q / t, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{n_seq} of {wl.batch} sequences (all {wl.num_q_heads} heads and {n_q} query token(s) "
                      f"each), append + decode step, mean of {reps} steps"}


def run_reference(args):
    """The reference arm: the CPU oracle, as it stands, on the host cores."""
    from paged_gqa_decode_02_gb300 import workloads as W
    from oracle import oracle

    dist, rank, world = _dist()
    if rank != 0:
        return
    wl = W.CONFIGS[args.workload]()
    n_seq = min(args.cpu_seqs, wl.batch)
    n_q = args.query_tokens
    qm = None if n_q == 1 else W.multi_token_queries(100, wl.batch, n_q, wl.num_q_heads, wl.head_dim)
    o, sub, rows = _oracle_setup(wl, n_seq, n_q)
    for _ in range(max(3, args.warmup)):
        _oracle_step(wl, o, sub, rows, n_q, qm)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        _oracle_step(wl, o, sub, rows, n_q, qm)
        times.append(time.perf_counter() - t0)
        if sum(times) > 120:
            break
    t = statistics.mean(times)
    v = n_seq * n_q / t
    res = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": world,
           "steps": len(times), "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64 (fp32 quantisation steps)",
           "data": "synthetic (same seeded workload)",
           "config": {"workload": WORKLOAD_TEXT[args.workload], "name": args.workload, "query_tokens": n_q},
           "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
                            "sample": f"{n_seq} of {wl.batch} sequences per step (all heads, {n_q} query "
                                      f"token(s) each), append + decode"},
           "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="qwen25_7b_bf16", choices=sorted(WORKLOAD_TEXT))
    ap.add_argument("--splits", type=int, default=0)
    ap.add_argument("--path", default="auto", choices=["auto", "cuda_core", "tensor_core"])
    ap.add_argument("--combine", default="separate", choices=["fused", "separate"])
    ap.add_argument("--unit-cost", type=int, default=-1,
                    help="phantom pages per unit in the cost-balanced partition (-1: the library default)")
    ap.add_argument("--no-early-plan", action="store_true",
                    help="decode plans only after the append kernel has finished")
    ap.add_argument("--cpu-seqs", type=int, default=1 << 30)
    ap.add_argument("--query-tokens", type=int, default=1,
                    help="causal query tokens per sequence (chunked prefill / speculative verification)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
