"""Python handle on the CPU oracle (pa_oracle.c) -- TEST INFRASTRUCTURE ONLY.

Only the tests, the package smoke check and the benchmark's CPU-baseline leg
use this module. It compiles pa_oracle.c with gcc (no CUDA, no code shared
with the CUDA library) and exposes:

  quant_channel(vals, L)           the per-channel asymmetric quantiser
  quant_channel_fp8(vals)          the per-channel symmetric E4M3 quantiser
  e4m3_encode(y), e4m3_value(c)    the E4M3 encoding and its values
  OraclePool                       a host copy of a paged KV pool in the
                                   library's storage format, with append(),
                                   decode() and decode_multi() (several
                                   causal query tokens per sequence)

See pa_oracle.c for the cited definitions and the readings taken where the
source pages are silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

KV_CODES = {"bf16": 0, "uint8": 1, "uint4": 2, "fp8": 3}


def build(force: bool = False) -> str:
    """Compile the oracle into oracle/_build/liboracle.so (gcc, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def build_variant(source_text: str, out_path: str) -> str:
    """Compile an edited copy of the oracle source (used by the mutation
    tests, which plant mistakes in the oracle to show the pins catch them)."""
    src = out_path + ".c"
    with open(src, "w") as f:
        f.write(source_text)
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
                    "-fPIC", "-shared", src, "-o", out_path, "-lm"], check=True)
    return out_path


def lib():
    """The oracle library; PA_ORACLE_LIB selects a planted-mistake build."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(os.environ.get("PA_ORACLE_LIB") or build())
            P = ctypes.c_void_p
            i32 = ctypes.c_int
            _lib.oracle_quant_channel.argtypes = [P, i32, i32, P, P, P]
            _lib.oracle_quant_channel.restype = None
            _lib.oracle_append.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, P, P, P, P, i32, i32]
            _lib.oracle_append.restype = i32
            _lib.oracle_decode.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, P, P, P, P, P,
                                           i32, P, P, i32, ctypes.c_double, P, ctypes.c_int64, P]
            _lib.oracle_decode.restype = i32
            _lib.oracle_decode_multi.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, P, P, P, P, P,
                                                 i32, i32, P, P, i32, ctypes.c_double, P,
                                                 ctypes.c_int64, P]
            _lib.oracle_decode_multi.restype = i32
            _lib.oracle_quant_channel_fp8.argtypes = [P, i32, P, P]
            _lib.oracle_quant_channel_fp8.restype = None
            _lib.oracle_e4m3_encode_array.argtypes = [P, ctypes.c_int64, P]
            _lib.oracle_e4m3_encode_array.restype = None
            _lib.oracle_e4m3_value.argtypes = [i32]
            _lib.oracle_e4m3_value.restype = ctypes.c_double
            _lib.oracle_num_threads.argtypes = []
            _lib.oracle_num_threads.restype = i32
            _lib.oracle_set_num_threads.argtypes = [i32]
            _lib.oracle_set_num_threads.restype = None
        return _lib


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Threads the oracle's parallel loops use from now on (timing only)."""
    lib().oracle_set_num_threads(int(n))


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def quant_channel(vals, L: int):
    """(scale float32, zp int, codes int32[n]) for one channel of one block."""
    v = np.ascontiguousarray(vals, dtype=np.float32)
    assert v.ndim == 1 and v.size >= 1
    sc = np.zeros(1, np.float32)
    zp = np.zeros(1, np.int32)
    codes = np.zeros(v.size, np.int32)
    lib().oracle_quant_channel(_p(v), v.size, int(L), _p(sc), _p(zp), _p(codes))
    return sc[0], int(zp[0]), codes


def quant_channel_fp8(vals):
    """(scale float32, codes int32[n] holding E4M3 bits) for one channel of one block."""
    v = np.ascontiguousarray(vals, dtype=np.float32)
    assert v.ndim == 1 and v.size >= 1
    sc = np.zeros(1, np.float32)
    codes = np.zeros(v.size, np.int32)
    lib().oracle_quant_channel_fp8(_p(v), v.size, _p(sc), _p(codes))
    return sc[0], codes


def e4m3_encode(y):
    """E4M3 bit patterns (uint8) of finite float32 values."""
    y = np.ascontiguousarray(y, dtype=np.float32)
    out = np.zeros(y.shape, np.uint8)
    lib().oracle_e4m3_encode_array(_p(y), y.size, _p(out))
    return out


def e4m3_value(codes):
    """float64 values of E4M3 bit patterns (NaN for the two NaN codes)."""
    c = np.asarray(codes).astype(np.int64)
    return np.array([lib().oracle_e4m3_value(int(x)) for x in c.ravel()], np.float64).reshape(c.shape)


class OraclePool:
    """Host copy of a paged KV pool, in the library's storage format.

    bf16 : k16/v16   uint16 [P, Hkv, bs, D]
    uint8: kc/vc     uint8  [P, Hkv, bs, D]
    uint4: kc/vc     uint8  [P, Hkv, bs, D/2]  (low nibble = even channel)
    fp8  : kc/vc     uint8  [P, Hkv, bs, D]    (E4M3 bits)
    quantised pools also hold ks/vs float32 [P, Hkv, D], and the integer ones
    kz/vz int32 [P, Hkv, D].
    """

    def __init__(self, kv_dtype, num_blocks, num_kv_heads, block_size, head_dim, fill=0):
        self.kv_dtype, self.P, self.Hkv, self.bs, self.D = (kv_dtype, int(num_blocks),
                                                            int(num_kv_heads), int(block_size),
                                                            int(head_dim))
        shp = (self.P, self.Hkv, self.bs, self.D)
        self.k16 = self.v16 = self.kc = self.vc = None
        self.ks = self.vs = self.kz = self.vz = None
        if kv_dtype == "bf16":
            self.k16 = np.full(shp, fill, np.uint16)
            self.v16 = np.full(shp, fill, np.uint16)
        else:
            w = self.D // 2 if kv_dtype == "uint4" else self.D
            self.kc = np.full(shp[:3] + (w,), fill, np.uint8)
            self.vc = np.full(shp[:3] + (w,), fill, np.uint8)
            self.ks = np.ones((self.P, self.Hkv, self.D), np.float32)
            self.vs = np.ones((self.P, self.Hkv, self.D), np.float32)
            if kv_dtype != "fp8":
                self.kz = np.zeros((self.P, self.Hkv, self.D), np.int32)
                self.vz = np.zeros((self.P, self.Hkv, self.D), np.int32)

    def append(self, k_bits, v_bits, cu_new, ctx_lens, block_table) -> int:
        k_bits = np.ascontiguousarray(k_bits, np.uint16)
        v_bits = np.ascontiguousarray(v_bits, np.uint16)
        cu_new = np.ascontiguousarray(cu_new, np.int32)
        ctx_lens = np.ascontiguousarray(ctx_lens, np.int32)
        block_table = np.ascontiguousarray(block_table, np.int32)
        B = ctx_lens.shape[0]
        MB = block_table.shape[1] if block_table.ndim == 2 else 0
        code = KV_CODES[self.kv_dtype]
        st = 0
        for new, p16, c, s, z in ((k_bits, self.k16, self.kc, self.ks, self.kz),
                                  (v_bits, self.v16, self.vc, self.vs, self.vz)):
            st = min(st, lib().oracle_append(code, self.P, self.Hkv, self.bs, self.D, _p(p16),
                                             _p(c), _p(s), _p(z), _p(new), _p(cu_new),
                                             _p(ctx_lens), _p(block_table), B, MB))
        return st

    def append_call(self, call) -> int:
        return self.append(call.k_bits, call.v_bits, call.cu_new, call.ctx_lens, call.block_table)

    def decode(self, q_bits, block_table, seq_lens, softmax_scale, rows=None):
        """fp64 attention output for the given flat rows (b * Hq + h); all rows
        when rows is None. Returns (out float64 [n_rows, D], status)."""
        q_bits = np.ascontiguousarray(q_bits, np.uint16)
        B, Hq, D = q_bits.shape
        assert D == self.D
        block_table = np.ascontiguousarray(block_table, np.int32)
        seq_lens = np.ascontiguousarray(seq_lens, np.int32)
        if rows is None:
            rows = np.arange(B * Hq, dtype=np.int64)
        rows = np.ascontiguousarray(rows, np.int64)
        out = np.zeros((rows.size, D), np.float64)
        st = lib().oracle_decode(KV_CODES[self.kv_dtype], self.P, self.Hkv, self.bs, self.D,
                                 _p(self.k16), _p(self.v16), _p(self.kc), _p(self.vc),
                                 _p(self.ks), _p(self.kz), _p(self.vs), _p(self.vz),
                                 _p(q_bits), Hq, _p(block_table), _p(seq_lens),
                                 block_table.shape[1], float(softmax_scale), _p(rows),
                                 rows.size, _p(out))
        return out, int(st)

    def decode_multi(self, q_bits, block_table, seq_lens, softmax_scale, rows=None):
        """Several query tokens per sequence, causal over the stored cache.
        q_bits is [B, n_q, Hq, D]; query token i of sequence b sees the first
        seq_lens[b] - (n_q - 1 - i) tokens. Rows are flat indices
        ((b * n_q) + i) * Hq + h (all when None). Returns (out float64
        [n_rows, D], status)."""
        q_bits = np.ascontiguousarray(q_bits, np.uint16)
        B, n_q, Hq, D = q_bits.shape
        assert D == self.D
        block_table = np.ascontiguousarray(block_table, np.int32)
        seq_lens = np.ascontiguousarray(seq_lens, np.int32)
        if rows is None:
            rows = np.arange(B * n_q * Hq, dtype=np.int64)
        rows = np.ascontiguousarray(rows, np.int64)
        out = np.zeros((rows.size, D), np.float64)
        st = lib().oracle_decode_multi(KV_CODES[self.kv_dtype], self.P, self.Hkv, self.bs, self.D,
                                       _p(self.k16), _p(self.v16), _p(self.kc), _p(self.vc),
                                       _p(self.ks), _p(self.kz), _p(self.vs), _p(self.vz),
                                       _p(q_bits), n_q, Hq, _p(block_table), _p(seq_lens),
                                       block_table.shape[1], float(softmax_scale), _p(rows),
                                       rows.size, _p(out))
        return out, int(st)
