"""Benchmark: one decode step of paged GQA attention per step -- append the
step's new token of every sequence (kv_quant_append), then attend
(paged_gqa_decode + split-KV combine) -- on the Qwen2.5-7B-shaped workload
(batch 32, 28 Q / 4 KV heads, head_dim 128, block 16, seq_lens U[512, 4096],
bf16 KV), synthetic seeded data. The same run measures the other workloads
(Qwen3-8B-shaped uint8 and fp8 KV, long-context uint4, prefix-sharing mix)
under "per_config".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--splits S] [--no-per-config]

Prints one JSON line. value = decode tokens per second (batch / step time),
whole job over all ranks. Two timings of each workload:
  isolated      every step (and every decode call) bracketed by its own CUDA
                events, with the L2 cache flushed (a 256 MiB write) before it,
                outside the brackets; `value`, `ms_per_step` and `roofline`
                come from these;
  back_to_back  K steps (calls) in one pair of events, each reading another
                of several copies of the pool (every copy larger than L2), as
                a decoding loop issues them.
`stream_ceiling` times the simplest read of the same number of bytes both ways
(pa_stream_read): what the launch, ramp-up and drain of one kernel cost at
this size.

With --gpus N > 1 and no torchrun environment the script starts N local
ranks itself (torch.distributed.run, 127.0.0.1). Every rank runs its own
replica of the workload on its own GPU (the path needs no exchange between
GPUs): weak scaling; times are the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import platform
import re
import socket
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
# measured in the same run as the headline workload
PER_CONFIG = ("qwen3_8b_int8", "long_uint4", "prefix_mix", "qwen3_8b_fp8")
L2_BYTES = 129 * 1000 * 1000
L2_TEXT = ("GPU arm, isolated: L2 flushed before every timed step and call (a 256 MiB write, outside the event "
           "brackets); GPU arm, back_to_back: inputs larger than L2 (each call reads another of {n} pool copies "
           "of {mb:.0f} MB); CPU arm: host memory")


def pool_copies(nbytes):
    """Pool copies the back-to-back timing rotates through: enough that every
    call reads memory that the calls before it pushed out of L2."""
    return max(2, -(-3 * L2_BYTES // max(int(nbytes), 1)))


PROFILE_FOR = {"qwen25_7b_bf16": "profiles/paged_gqa_decode_qwen25_7b_bf16.md",
               "qwen3_8b_int8": "profiles/paged_gqa_decode_qwen3_8b_int8.md",
               "long_uint4": "profiles/paged_gqa_decode_long_uint4.md",
               "prefix_mix": "profiles/paged_gqa_decode_prefix_mix.md",
               "qwen3_8b_fp8": "profiles/paged_gqa_decode_qwen3_8b_fp8.md"}


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


def _cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform.processor() or platform.machine()


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


def workload_config(wl, name, n_q, world=1):
    """The workload's description, the same for both arms of the benchmark."""
    from paged_gqa_decode_02_gb300.metrics import decode_bytes
    nb = decode_bytes(wl, n_q)
    cfg = {"workload": WORKLOAD_TEXT[name], "name": name, "batch": wl.batch, "num_q_heads": wl.num_q_heads,
           "num_kv_heads": wl.num_kv_heads, "head_dim": wl.head_dim, "block_size": wl.block_size,
           "kv_dtype": wl.kv_dtype, "tokens_cached": nb["tokens_scanned"], "query_tokens": n_q,
           "step": (f"append {n_q} token(s)/seq (kv_quant_append) + paged_gqa_decode"
                    + (f" with {n_q} causal query tokens per sequence" if n_q > 1 else "")
                    + " + split-KV combine"),
           "l2": L2_TEXT.format(n=pool_copies(nb["algorithmic"]), mb=nb["algorithmic"] / 1e6),
           "parallelism": f"replicas x{world} (no exchange)"}
    return cfg, nb


class WorkloadRun:
    """One workload on one GPU: `n_rot` identical pools (the copies that the
    back-to-back timing rotates through), the step's inputs, and timers."""

    def __init__(self, name, args, dev, n_q=1, n_rot=None):
        import torch
        from paged_gqa_decode_02_gb300 import workloads as W
        from paged_gqa_decode_02_gb300.binding import PagedKVPool
        self.torch = torch
        self.name, self.args, self.dev, self.n_q = name, args, dev, n_q
        wl = self.wl = W.CONFIGS[name]()
        self.cfg, self.nb = workload_config(wl, name, n_q, int(os.environ.get("WORLD_SIZE", "1")))
        self.n_rot = n_rot or pool_copies(self.nb["algorithmic"])
        fills = [(self.d(c.k_bits), self.d(c.v_bits), self.d(c.cu_new), self.d(c.ctx_lens),
                  self.d(c.block_table), c.max_new) for c in wl.fill_calls(leave_last=(n_q == 1))]
        self.pools = []
        for _ in range(self.n_rot):
            p = PagedKVPool(wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim, wl.kv_dtype, dev.index)
            p.set_decode_path(args.path, fused_combine=(args.combine == "fused"), early_plan=not args.no_early_plan)
            p.set_unit_cost(args.unit_cost)
            for k, v, cu, ctx, tb, mn in fills:
                p.append_kv(k, v, cu, ctx, tb, max_new_per_seq=mn)
            self.pools.append(p)
        del fills
        step = self.step = wl.step_call(n_q)
        self.st = (self.d(step.k_bits), self.d(step.v_bits), self.d(step.cu_new), self.d(step.ctx_lens))
        if n_q == 1:  # the same new tokens as rows [B][Hkv][D], for the fused decode step
            kr = np.zeros((wl.batch, wl.num_kv_heads, wl.head_dim), np.uint16)
            vr = np.zeros_like(kr)
            for b in range(wl.batch):
                if step.cu_new[b + 1] > step.cu_new[b]:
                    kr[b], vr[b] = step.k_bits[step.cu_new[b]], step.v_bits[step.cu_new[b]]
            self.rows = (self.d(kr), self.d(vr))
        B, Hq, D = wl.batch, wl.num_q_heads, wl.head_dim
        self.q_bits = wl.q_bits if n_q == 1 else W.multi_token_queries(100, B, n_q, Hq, D)
        self.table, self.lens, self.q = self.d(wl.block_table), self.d(wl.seq_lens), self.d(self.q_bits)
        self.outs = [torch.empty(self.q_bits.shape, dtype=torch.float32, device=dev) for _ in range(self.n_rot)]
        self.ws = [p.workspace(B, Hq, args.splits) for p in self.pools]
        self.splits_used = self.pools[0].num_splits(args.splits)
        self.flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
        self.stream = torch.cuda.current_stream(dev)

    def d(self, a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        return self.torch.from_numpy(a).to(self.dev)

    def decode_call(self, i, q=None, table=None, lens=None):
        q = self.q if q is None else q
        table = self.table if table is None else table
        lens = self.lens if lens is None else lens
        p, out = self.pools[i], self.outs[i]
        if self.n_q == 1:
            p.decode(q, table, lens, self.wl.softmax_scale, out=out, workspace=self.ws[i],
                     num_splits=self.args.splits)
        else:
            p.decode_multi(q, table, lens, self.wl.softmax_scale, out=out, num_splits=self.args.splits)

    def step_call(self, i):
        # append then decode back to back, as a decode loop runs them (the
        # decode's planning may overlap the append; see --no-early-plan)
        k, v, cu, ctx = self.st
        self.pools[i].append_kv(k, v, cu, ctx, self.table, max_new_per_seq=self.n_q)
        self.decode_call(i)

    def fused_step_call(self, i):
        # the decode step in one decode launch (pa_decode_step)
        self.pools[i].decode_step(self.rows[0], self.rows[1], self.q, self.table, self.lens, self.wl.softmax_scale,
                                  out=self.outs[i], workspace=self.ws[i], num_splits=self.args.splits)

    def isolated(self, fn, K):
        torch = self.torch
        e0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        e1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        for i in range(K):
            self.flush.fill_(1)
            e0[i].record(self.stream)
            fn(0)
            e1[i].record(self.stream)
        torch.cuda.synchronize()
        return [e0[i].elapsed_time(e1[i]) for i in range(K)]

    def back_to_back(self, fn, K):
        torch = self.torch
        for i in range(self.n_rot):
            fn(i)
        a = torch.cuda.Event(enable_timing=True)
        z = torch.cuda.Event(enable_timing=True)
        a.record(self.stream)
        for i in range(K):
            fn(i % self.n_rot)
        z.record(self.stream)
        torch.cuda.synchronize()
        return a.elapsed_time(z) / K

    def e2e(self, K):
        """The step through the public API from pinned host memory: H2D of the
        step's inputs, append, decode, D2H of the output, all in the region.
        The inputs (new K/V, their offsets and context lengths, the block
        table, the lengths, q) are staged in one pinned buffer, each at a
        256-byte offset, and go over in one copy; the API is called on device
        views of the copied buffer."""
        torch = self.torch
        s = self.step
        arrays = [(k, np.ascontiguousarray(v).view(np.int16) if v.dtype == np.uint16 else np.ascontiguousarray(v))
                  for k, v in (("k", s.k_bits), ("v", s.v_bits), ("cu", s.cu_new), ("ctx", s.ctx_lens),
                               ("table", self.wl.block_table), ("lens", self.wl.seq_lens), ("q", self.q_bits))]
        offs, total = {}, 0
        for k, a in arrays:
            offs[k] = total
            total += (a.nbytes + 255) // 256 * 256
        h_buf = torch.zeros(total, dtype=torch.uint8).pin_memory()
        for k, a in arrays:
            h_buf[offs[k]:offs[k] + a.nbytes].copy_(torch.from_numpy(a.reshape(-1).view(np.uint8)))
        d_buf = torch.empty(total, dtype=torch.uint8, device=self.dev)
        tdt = {np.dtype(np.int16): torch.int16, np.dtype(np.int32): torch.int32}
        d_in = {k: d_buf[offs[k]:offs[k] + a.nbytes].view(tdt[a.dtype]).view(a.shape) for k, a in arrays}
        h_out = torch.empty(self.q_bits.shape, dtype=torch.float32).pin_memory()
        bi = total
        bo = h_out.numel() * h_out.element_size()
        ms = []
        for i in range(K + 3):
            self.flush.fill_(1)
            a = torch.cuda.Event(enable_timing=True)
            z = torch.cuda.Event(enable_timing=True)
            a.record(self.stream)
            d_buf.copy_(h_buf, non_blocking=True)
            self.pools[0].append_kv(d_in["k"], d_in["v"], d_in["cu"], d_in["ctx"], d_in["table"],
                                    max_new_per_seq=self.n_q)
            self.decode_call(0, d_in["q"], d_in["table"], d_in["lens"])
            h_out.copy_(self.outs[0], non_blocking=True)
            z.record(self.stream)
            z.synchronize()
            if i >= 3:
                ms.append(a.elapsed_time(z))
        return statistics.mean(ms), bi, bo

    def device_error(self):
        for p in self.pools:
            st, flags = p.device_error()
            if st != 0 or flags != 0:
                return st, flags
        return 0, 0

    def close(self):
        for p in self.pools:
            p.close()
        self.pools = []


def measure(run, dist, world, K, warmup, peak, peak_kind, K_e2e):
    """All timings of one workload (max over ranks); the JSON fields."""
    B, n_q = run.wl.batch, run.n_q
    for _ in range(max(3, warmup)):
        run.flush.fill_(1)
        run.step_call(0)
    run.torch.cuda.synchronize()
    st, flags = run.device_error()
    assert st == 0 and flags == 0, f"device error word {flags:#x} during warm-up ({run.name})"
    _barrier(dist)
    step_ms = run.isolated(run.step_call, K)
    dec_ms = run.isolated(run.decode_call, K)
    b2b_step = run.back_to_back(run.step_call, K)
    b2b_dec = run.back_to_back(run.decode_call, K)
    fused_ms = run.isolated(run.fused_step_call, K) if n_q == 1 else None
    st, flags = run.device_error()
    assert st == 0 and flags == 0, f"device error word {flags:#x} during timing ({run.name})"
    t_step = _max_over_ranks(dist, statistics.mean(step_ms) / 1e3)
    t_dec = _max_over_ranks(dist, statistics.mean(dec_ms) / 1e3)
    t_b2b_step = _max_over_ranks(dist, b2b_step / 1e3)
    t_b2b_dec = _max_over_ranks(dist, b2b_dec / 1e3)
    e2e_ms, bi, bo = run.e2e(K_e2e)
    t_e2e = _max_over_ranks(dist, e2e_ms / 1e3)
    alg = run.nb["algorithmic"]
    ach = alg / t_dec / 1e9
    ach_b2b = alg / t_b2b_dec / 1e9
    return {
        "value": world * B * n_q / t_step,
        "ms_per_step": t_step * 1e3,
        "decode_us": t_dec * 1e6,
        "median_us": {"step": statistics.median(step_ms) * 1e3, "decode": statistics.median(dec_ms) * 1e3},
        "hbm_gbs": ach,
        "kv_tokens_per_s": world * run.nb["tokens_scanned"] / t_dec,
        "roofline": {"bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s", "frac": ach / peak,
                     "traffic": _traffic(run.name, run.args.path) if n_q == 1 else None,
                     "peak_kind": f"{peak_kind} (copy bandwidth, MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "algorithmic_bytes_per_launch": alg,
                     "timed": "pa_decode call (decode kernel + split-KV combine) alone, isolated: CUDA events "
                              "on the launch stream around each call, L2 flushed before it"},
        "back_to_back": {"step_us": t_b2b_step * 1e6, "decode_us": t_b2b_dec * 1e6,
                         "tokens_per_s": world * B * n_q / t_b2b_step,
                         "decode_gbs": ach_b2b, "decode_frac": ach_b2b / peak, "pool_copies": run.n_rot},
        "e2e": {"value": world * B * n_q / t_e2e, "unit": "tokens/s", "h2d_bytes_per_step": bi,
                "d2h_bytes_per_step": bo},
        "fused_step_us": None if fused_ms is None else {
            "isolated": _max_over_ranks(dist, statistics.mean(fused_ms) / 1e3) * 1e6,
            "note": "pa_decode_step (store the new tokens and attend in one decode launch + combine), timed "
                    "like the step above; the step (pa_append_kv then pa_decode) is what value reports"},
        "launch": {"num_splits": run.splits_used, "decode_path": run.args.path,
                   "combine": run.args.combine if n_q == 1 else "separate", "early_plan": not run.args.no_early_plan,
                   "unit_cost": run.args.unit_cost},
    }


def stream_ceiling(dev, nbytes, K):
    """The simplest kernel that reads `nbytes` (the library's calibration read,
    pa_stream_read: 16-byte streaming loads over every SM), timed like the
    decode call: isolated with the L2 flushed, and back to back over three
    copies. What one kernel's launch, ramp-up and drain cost at this size."""
    import torch
    from paged_gqa_decode_02_gb300 import binding
    n = max(16, (nbytes + 15) // 16 * 16)
    bufs = [torch.ones(n // 4, dtype=torch.float32, device=dev) for _ in range(3)]
    sink = torch.zeros(4, dtype=torch.int32, device=dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    for b in bufs:
        binding.pa_stream_read(b, sink)
    ev = []
    for i in range(K):
        flush.fill_(1)
        a = torch.cuda.Event(enable_timing=True)
        z = torch.cuda.Event(enable_timing=True)
        a.record()
        binding.pa_stream_read(bufs[0], sink)
        z.record()
        ev.append((a, z))
    torch.cuda.synchronize()
    iso = statistics.mean(a.elapsed_time(z) for a, z in ev) / 1e3
    a = torch.cuda.Event(enable_timing=True)
    z = torch.cuda.Event(enable_timing=True)
    a.record()
    for i in range(K):
        binding.pa_stream_read(bufs[i % 3], sink)
    z.record()
    torch.cuda.synchronize()
    b2b = a.elapsed_time(z) / K / 1e3
    return {"bytes": n, "isolated_us": iso * 1e6, "isolated_gbs": n / iso / 1e9,
            "back_to_back_us": b2b * 1e6, "back_to_back_gbs": n / b2b / 1e9,
            "kernel": "pa_stream_read: 16-byte streaming loads over every SM, nothing else (a read of the same bytes)"}


def run_ours(args):
    import torch
    from paged_gqa_decode_02_gb300 import build as pbuild

    dist, rank, world = _dist()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if rank == 0:
        pbuild.build()
    _barrier(dist)
    dev = torch.device("cuda", local)
    peak, peak_kind = _peaks()
    K = args.steps
    n_q = args.query_tokens

    run = WorkloadRun(args.workload, args, dev, n_q)
    clocks = ClockSampler(local)
    clocks.start()
    # soak so that the clock record covers a loaded GPU before and during timing
    t_end = time.time() + 1.0
    while time.time() < t_end:
        run.flush.fill_(1)
        run.step_call(0)
    torch.cuda.synchronize()
    head = measure(run, dist, world, K, args.warmup, peak, peak_kind, max(10, min(K, 200)))
    ceiling = stream_ceiling(dev, run.nb["algorithmic"], min(K, 500))
    clk = clocks.stop()
    cfg = dict(run.cfg)
    res = {
        "metric": METRIC,
        "value": head["value"],
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": head["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if run.wl.kv_dtype == "bf16" else f"{run.wl.kv_dtype} codes, fp32 math",
        "data": "synthetic (seeded N(0,1) bf16 q/K/V, block tables from a seeded permutation)",
        "config": cfg,
    }
    res.update({k: v for k, v in head.items() if k not in ("value", "ms_per_step")})
    res["stream_ceiling"] = ceiling
    res["gpu_launches"] = 3 * K
    res["gpu_launches_note"] = "3 per step in the isolated step timing: kv_append_kernel, " \
                               "paged_gqa_decode_kernel, splitkv_combine_kernel"
    res["clocks"] = clk
    run.close()
    del run
    torch.cuda.empty_cache()

    if not args.no_per_config and n_q == 1:
        per = {}
        Kp = max(3, min(K, 300))
        pclk = ClockSampler(local)
        pclk.start()
        for name in PER_CONFIG:
            if name == args.workload:
                continue
            r = WorkloadRun(name, args, dev, 1)
            m = measure(r, dist, world, Kp, args.warmup, peak, peak_kind, max(10, min(Kp, 100)))
            m["config"] = dict(r.cfg)
            m["steps"] = Kp
            m["dtype"] = "bf16" if r.wl.kv_dtype == "bf16" else f"{r.wl.kv_dtype} codes, fp32 math"
            if name == "prefix_mix":
                m["logical_bytes"] = r.nb["logical"]
                m["effective_gbs"] = r.nb["logical"] / (m["decode_us"] / 1e6) / 1e9
            per[name] = m
            r.close()
            del r
            torch.cuda.empty_cache()
        res["per_config"] = per
        res["per_config_clocks"] = pclk.stop()
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_seqs, n_q)
    if rank == 0:
        print(json.dumps(res), flush=True)


def profile_run(args):
    """W warm-up steps, then K isolated steps of one pool: per step the L2
    flush (torch fill), kv_append_kernel, paged_gqa_decode_kernel and
    splitkv_combine_kernel, and nothing else."""
    import torch
    from paged_gqa_decode_02_gb300 import build as pbuild
    pbuild.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(0)
    run = WorkloadRun(args.workload, args, dev, args.query_tokens, n_rot=1)
    for _ in range(max(3, args.warmup)):
        run.flush.fill_(1)
        run.step_call(0)
    ms = run.isolated(run.step_call, args.steps)
    st, flags = run.device_error()
    assert st == 0 and flags == 0, f"device error word {flags:#x}"
    print(json.dumps({"profile_run": args.workload, "steps": args.steps, "warmup": args.warmup,
                      "step_us_mean": statistics.mean(ms) * 1e3}), flush=True)
    run.close()


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


def _oracle_append(o, sub):
    assert o.append(*sub) == 0


def _oracle_decode(wl, o, rows, n_q=1, q_multi=None):
    if n_q == 1:
        out, st = o.decode(wl.q_bits, wl.block_table, wl.seq_lens, wl.softmax_scale, rows=rows)
    else:
        out, st = o.decode_multi(q_multi, wl.block_table, wl.seq_lens, wl.softmax_scale, rows=rows)
    assert st == 0
    return out


def _sample_bytes(wl, n_seq, n_q):
    """Algorithmic bytes of the decode restricted to the first n_seq sequences."""
    from paged_gqa_decode_02_gb300.metrics import decode_bytes

    class _Sub:
        pass
    s = _Sub()
    s.batch, s.num_q_heads, s.num_kv_heads = n_seq, wl.num_q_heads, wl.num_kv_heads
    s.head_dim, s.block_size, s.kv_dtype = wl.head_dim, wl.block_size, wl.kv_dtype
    s.seq_lens, s.block_table = wl.seq_lens[:n_seq], wl.block_table[:n_seq]
    return decode_bytes(s, n_q)["algorithmic"]


def _time_oracle(wl, o, sub, rows, n_q, qm, budget_s, max_reps):
    """Mean append and decode times of the oracle over up to max_reps steps."""
    _oracle_append(o, sub)
    _oracle_decode(wl, o, rows, n_q, qm)
    t_app, t_dec, reps, t0 = 0.0, 0.0, 0, time.perf_counter()
    while True:
        a = time.perf_counter()
        _oracle_append(o, sub)
        b = time.perf_counter()
        _oracle_decode(wl, o, rows, n_q, qm)
        c = time.perf_counter()
        t_app += b - a
        t_dec += c - b
        reps += 1
        if c - t0 > budget_s or reps >= max_reps:
            break
    return t_app / reps, t_dec / reps, reps


def cpu_baseline(name, n_seq, n_q=1):
    """The oracle (fp64, scalar C) on this host's cores: all of them, and one."""
    from oracle import oracle
    from paged_gqa_decode_02_gb300 import workloads as W
    wl = W.CONFIGS[name]()
    n_seq = min(n_seq, wl.batch)
    o, sub, rows = _oracle_setup(wl, n_seq, n_q)
    qm = None if n_q == 1 else W.multi_token_queries(100, wl.batch, n_q, wl.num_q_heads, wl.head_dim)
    cores = oracle.num_threads()
    ta, td, reps = _time_oracle(wl, o, sub, rows, n_q, qm, 8.0, 20)
    # one thread: a smaller sample (a quarter of the sequences, at least one)
    n1 = max(1, n_seq // 4)
    o1, sub1, rows1 = _oracle_setup(wl, n1, n_q)
    oracle.set_num_threads(1)
    try:
        ta1, td1, reps1 = _time_oracle(wl, o1, sub1, rows1, n_q, qm, 8.0, 5)
    finally:
        oracle.set_num_threads(cores)
    nbytes = _sample_bytes(wl, n_seq, n_q)
    nbytes1 = _sample_bytes(wl, n1, n_q)
    return {"value": n_seq * n_q / (ta + td), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "cpu_model": _cpu_model(),
            "append_ms": ta * 1e3, "decode_ms": td * 1e3, "decode_gbs": nbytes / td / 1e9,
            "single_thread": {"value": n1 * n_q / (ta1 + td1), "unit": "tokens/s", "cores": 1,
                              "append_ms": ta1 * 1e3, "decode_ms": td1 * 1e3, "decode_gbs": nbytes1 / td1 / 1e9,
                              "sample": f"{n1} of {wl.batch} sequences, mean of {reps1} steps"},
            "sample": f"{n_seq} of {wl.batch} sequences (all {wl.num_q_heads} heads and {n_q} query token(s) "
                      f"each), append + decode step, mean of {reps} steps; GB/s over the sample's "
                      f"algorithmic bytes ({nbytes / 1e6:.1f} MB)"}


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
        _oracle_append(o, sub)
        _oracle_decode(wl, o, rows, n_q, qm)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        _oracle_append(o, sub)
        _oracle_decode(wl, o, rows, n_q, qm)
        times.append(time.perf_counter() - t0)
        if sum(times) > 120:
            break
    t = statistics.mean(times)
    v = n_seq * n_q / t
    cfg, _ = workload_config(wl, args.workload, n_q, world)
    res = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": world,
           "steps": len(times), "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64 (fp32 quantisation steps)",
           "data": "synthetic (same seeded workload)", "config": cfg,
           "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
                            "cpu_model": _cpu_model(),
                            "sample": f"{n_seq} of {wl.batch} sequences per step (all heads, {n_q} query "
                                      f"token(s) each), append + decode"},
           "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _launch_ranks(n):
    """Start n local ranks of this script (one per GPU) and pass their output
    through; rank 0 prints the JSON line."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", str(n),
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), os.path.abspath(__file__)] + sys.argv[1:]
    return subprocess.run(cmd, cwd=ROOT).returncode


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
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
    ap.add_argument("--no-per-config", action="store_true",
                    help="measure the headline workload only")
    ap.add_argument("--profile-run", action="store_true",
                    help="only W warm-up and K isolated steps of --workload (one pool, no other timings): "
                         "the short, fixed launch sequence that profiler captures use")
    args = ap.parse_args()
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(_launch_ranks(args.gpus))
    if args.impl == "reference":
        run_reference(args)
    elif args.profile_run:
        profile_run(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
