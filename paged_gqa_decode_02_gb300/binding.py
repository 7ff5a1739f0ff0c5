"""Thin ctypes binding of libpagedattn (include/pagedattn.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels. torch supplies device memory and streams. The functions keep the C
names (pa_create_pool, pa_append_kv, pa_decode, pa_destroy, ...); PagedKVPool
is a small convenience wrapper over them.

If the shared library is missing this module raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import numpy as np

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libpagedattn.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "pagedattn.h")

PA_KV_BF16, PA_KV_UINT8, PA_KV_UINT4, PA_KV_FP8 = 0, 1, 2, 3
KV_DTYPES = {"bf16": PA_KV_BF16, "uint8": PA_KV_UINT8, "uint4": PA_KV_UINT4, "fp8": PA_KV_FP8}
STATUS = {0: "PA_OK", 1: "PA_ERR_INVALID_ARG", 2: "PA_ERR_UNSUPPORTED", 3: "PA_ERR_OOM",
          4: "PA_ERR_CUDA", 5: "PA_ERR_DEVICE_BOUNDS", 6: "PA_ERR_TIMEOUT"}
DEVERR_BLOCK_TABLE, DEVERR_SEQ_LEN, DEVERR_APPEND, DEVERR_TIMEOUT = 0x1, 0x2, 0x4, 0x8
PA_SWAP_OUT, PA_SWAP_IN = 0, 1


class PagedAttnError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


class pa_pool_desc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32), ("device", ctypes.c_int32)]


class pa_pool_buffers(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("k_scale", ctypes.c_void_p),
                ("k_zp", ctypes.c_void_p), ("v_scale", ctypes.c_void_p), ("v_zp", ctypes.c_void_p),
                ("page_stride", ctypes.c_size_t), ("num_pages", ctypes.c_size_t)]


_lib = None
_lock = threading.Lock()


def header_symbols():
    """Function names declared in include/pagedattn.h."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:PA_API\s+)?(?:pa_status|size_t|int32_t|const char\*)\s+(pa_\w+)\s*\(",
                                 text, re.M)))


def lib():
    """Load libpagedattn.so (built by paged_gqa_decode_02_gb300.build)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run paged_gqa_decode_02_gb300.build.build() "
                               "(the CUDA library is required; there is no fallback)")
        L = ctypes.CDLL(LIB_PATH)
        P, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        L.pa_create_pool.argtypes = [ctypes.POINTER(pa_pool_desc), ctypes.POINTER(P)]
        L.pa_destroy.argtypes = [P]
        L.pa_append_kv.argtypes = [P, P, P, P, P, P, I32, I32, I32, P]
        L.pa_decode.argtypes = [P, P, P, P, I32, I32, I32, ctypes.c_float, P, P, SZ, I32, P]
        L.pa_decode_step.argtypes = [P, P, P, P, P, P, I32, I32, I32, ctypes.c_float, P, P, SZ, I32, P]
        L.pa_decode_workspace_bytes.argtypes = [P, I32, I32, I32]
        L.pa_decode_workspace_bytes.restype = SZ
        L.pa_decode_multi.argtypes = [P, P, P, P, I32, I32, I32, I32, ctypes.c_float, P, P, SZ, I32, P]
        L.pa_decode_multi_workspace_bytes.argtypes = [P, I32, I32, I32, I32]
        L.pa_decode_multi_workspace_bytes.restype = SZ
        L.pa_pool_set_decode_path.argtypes = [P, I32]
        L.pa_pool_set_decode_path.restype = I32
        L.pa_pool_set_unit_cost.argtypes = [P, I32]
        L.pa_pool_set_unit_cost.restype = I32
        I64, PI32 = ctypes.c_int64, ctypes.POINTER(ctypes.c_int32)
        L.pa_bm_create.argtypes = [I32, I32, I32, ctypes.POINTER(P)]
        L.pa_bm_create.restype = I32
        L.pa_bm_destroy.argtypes = [P]
        L.pa_bm_destroy.restype = I32
        L.pa_bm_add_sequence.argtypes = [P, I64, P, I32, PI32]
        L.pa_bm_add_sequence.restype = I32
        L.pa_bm_fork.argtypes = [P, I64, I64]
        L.pa_bm_fork.restype = I32
        L.pa_bm_append_tokens.argtypes = [P, I64, P, I32, PI32, PI32, I32, PI32]
        L.pa_bm_append_tokens.restype = I32
        L.pa_bm_free_sequence.argtypes = [P, I64]
        L.pa_bm_free_sequence.restype = I32
        L.pa_bm_block_table.argtypes = [P, I64, P, I32, PI32, ctypes.POINTER(I64)]
        L.pa_bm_block_table.restype = I32
        L.pa_bm_num_free_blocks.argtypes = [P]
        L.pa_bm_num_free_blocks.restype = I32
        L.pa_bm_ref_count.argtypes = [P, I32]
        L.pa_bm_ref_count.restype = I32
        L.pa_copy_blocks.argtypes = [P, P, P, I32, P]
        L.pa_copy_blocks.restype = I32
        L.pa_selftest_wait_timeout.argtypes = [I32, I64, ctypes.POINTER(ctypes.c_uint32)]
        L.pa_selftest_wait_timeout.restype = I32
        L.pa_stream_read.argtypes = [P, SZ, P, P]
        L.pa_stream_read.restype = I32
        L.pa_pool_block_bytes.argtypes = [P]
        L.pa_pool_block_bytes.restype = ctypes.c_size_t
        L.pa_swap_blocks.argtypes = [P, P, I32, P, P, I32, I32, P]
        L.pa_swap_blocks.restype = I32
        L.pa_bm_set_cpu_blocks.argtypes = [P, I32]
        L.pa_bm_set_cpu_blocks.restype = I32
        L.pa_bm_num_free_cpu_blocks.argtypes = [P]
        L.pa_bm_num_free_cpu_blocks.restype = I32
        L.pa_bm_swap_out.argtypes = [P, I64, P, P, I32, PI32]
        L.pa_bm_swap_out.restype = I32
        L.pa_bm_swap_in.argtypes = [P, I64, P, P, I32, PI32]
        L.pa_bm_swap_in.restype = I32
        L.pa_bm_swapped_slots.argtypes = [P, I64, P, I32, PI32]
        L.pa_bm_swapped_slots.restype = I32
        L.pa_decode_num_splits.argtypes = [P, I32]
        L.pa_decode_num_splits.restype = I32
        L.pa_pool_view.argtypes = [P, ctypes.POINTER(pa_pool_buffers)]
        L.pa_get_device_error.argtypes = [P, P, ctypes.POINTER(ctypes.c_uint32)]
        L.pa_status_string.argtypes = [I32]
        L.pa_status_string.restype = ctypes.c_char_p
        L.pa_last_error.argtypes = []
        L.pa_last_error.restype = ctypes.c_char_p
        for f in ("pa_create_pool", "pa_destroy", "pa_append_kv", "pa_decode", "pa_pool_view",
                  "pa_get_device_error"):
            getattr(L, f).restype = I32
        _lib = L
        return L


def _check(status):
    if status != 0:
        raise PagedAttnError(status, lib().pa_last_error().decode(errors="replace"))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


# ------------------------------------------------------------------ C-named entry points
def pa_create_pool(num_blocks, block_size, num_kv_heads, head_dim, kv_dtype, device=0):
    d = pa_pool_desc(int(num_blocks), int(block_size), int(num_kv_heads), int(head_dim),
                     KV_DTYPES[kv_dtype] if isinstance(kv_dtype, str) else int(kv_dtype), int(device))
    h = ctypes.c_void_p()
    _check(lib().pa_create_pool(ctypes.byref(d), ctypes.byref(h)))
    return h


def pa_destroy(handle):
    _check(lib().pa_destroy(handle))


def pa_append_kv(handle, k_new, v_new, cu_new, ctx_lens, block_table, batch, max_blocks,
                 max_new_per_seq=0, stream=None):
    _check(lib().pa_append_kv(handle, _ptr(k_new), _ptr(v_new), _ptr(cu_new), _ptr(ctx_lens),
                              _ptr(block_table), int(batch), int(max_blocks), int(max_new_per_seq),
                              _stream(stream)))


def pa_decode(handle, q, block_table, seq_lens, batch, num_q_heads, max_blocks, softmax_scale, out,
              workspace, workspace_bytes, num_splits=0, stream=None):
    _check(lib().pa_decode(handle, _ptr(q), _ptr(block_table), _ptr(seq_lens), int(batch),
                           int(num_q_heads), int(max_blocks), float(softmax_scale), _ptr(out),
                           _ptr(workspace), int(workspace_bytes), int(num_splits), _stream(stream)))


def pa_decode_workspace_bytes(handle, batch, num_q_heads, num_splits=0):
    return int(lib().pa_decode_workspace_bytes(handle, int(batch), int(num_q_heads), int(num_splits)))


PA_DECODE_AUTO, PA_DECODE_CUDA_CORE, PA_DECODE_TENSOR_CORE = 0, 1, 2
PA_DECODE_FUSED_COMBINE = 4
PA_DECODE_EARLY_PLAN = 8
DECODE_PATHS = {"auto": 0, "cuda_core": 1, "tensor_core": 2}


def pa_pool_set_decode_path(handle, path):
    _check(lib().pa_pool_set_decode_path(handle, DECODE_PATHS[path] if isinstance(path, str) else int(path)))


def pa_pool_set_unit_cost(handle, unit_cost_pages):
    _check(lib().pa_pool_set_unit_cost(handle, int(unit_cost_pages)))


def pa_decode_num_splits(handle, num_splits=0):
    return int(lib().pa_decode_num_splits(handle, int(num_splits)))


def pa_stream_read(src, sink, stream=None):
    """Bandwidth calibration: read the whole of tensor `src` (16-byte aligned,
    its size a multiple of 16 bytes) with the simplest streaming kernel; `sink`
    is a device int32 tensor. Asynchronous."""
    _check(lib().pa_stream_read(_ptr(src), src.numel() * src.element_size(), _ptr(sink), _stream(stream)))


def pa_get_device_error(handle, stream=None):
    flags = ctypes.c_uint32(0)
    st = lib().pa_get_device_error(handle, _stream(stream), ctypes.byref(flags))
    return st, int(flags.value)


class _DevArray:
    """Exposes a device address range to torch via __cuda_array_interface__."""

    def __init__(self, ptr, shape, typestr):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr,
                                         "data": (int(ptr), False), "version": 2, "strides": None}


def _view(ptr, shape, typestr, device):
    return torch.as_tensor(_DevArray(ptr, shape, typestr), device=device)


class PagedKVPool:
    """A paged KV pool on one GPU (owns a pa_pool handle)."""

    def __init__(self, num_blocks, block_size, num_kv_heads, head_dim, kv_dtype="bf16", device=0):
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)
        self.num_kv_heads, self.head_dim = int(num_kv_heads), int(head_dim)
        self.kv_dtype = kv_dtype
        self.device = torch.device("cuda", device) if isinstance(device, int) else torch.device(device)
        with torch.cuda.device(self.device):
            self.handle = pa_create_pool(num_blocks, block_size, num_kv_heads, head_dim, kv_dtype,
                                         self.device.index)
        self._ws = None

    def close(self):
        if self.handle is not None:
            pa_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def view(self):
        """torch tensors aliasing the pool's components (strided views over the
        page records, see pagedattn.h)."""
        b = pa_pool_buffers()
        _check(lib().pa_pool_view(self.handle, ctypes.byref(b)))
        P, H, bs, D = self.num_blocks, self.num_kv_heads, self.block_size, self.head_dim
        stride, n = int(b.page_stride), int(b.num_pages)
        rec = _view(b.k, (n * stride,), "|u1", self.device).view(P, H, stride)

        def comp(ptr, nbytes, dtype):
            off = int(ptr) - int(b.k)
            return rec[:, :, off:off + nbytes].view(dtype)

        if self.kv_dtype == "bf16":
            return {"k": comp(b.k, bs * D * 2, torch.int16).unflatten(2, (bs, D)),
                    "v": comp(b.v, bs * D * 2, torch.int16).unflatten(2, (bs, D))}
        w = D // 2 if self.kv_dtype == "uint4" else D
        parts = {"k": comp(b.k, bs * w, torch.uint8).unflatten(2, (bs, w)),
                 "v": comp(b.v, bs * w, torch.uint8).unflatten(2, (bs, w)),
                 "k_scale": comp(b.k_scale, D * 4, torch.float32),
                 "v_scale": comp(b.v_scale, D * 4, torch.float32)}
        if self.kv_dtype != "fp8":  # fp8 pools hold no zero points
            parts["k_zp"] = comp(b.k_zp, D * 4, torch.int32)
            parts["v_zp"] = comp(b.v_zp, D * 4, torch.int32)
        return parts

    def copy_blocks(self, src, dst, stream=None):
        """Copy whole blocks src[i] -> dst[i] (copy-on-write of shared blocks)."""
        s_ = np.ascontiguousarray(src, dtype=np.int32)
        d_ = np.ascontiguousarray(dst, dtype=np.int32)
        assert s_.size == d_.size
        st = stream if stream is not None else torch.cuda.current_stream(self.device).cuda_stream
        _check(lib().pa_copy_blocks(self.handle, s_.ctypes.data_as(ctypes.c_void_p), d_.ctypes.data_as(ctypes.c_void_p),
                                    int(s_.size), ctypes.c_void_p(st)))

    def block_bytes(self):
        """Bytes of one block's page records (a slot of the host swap tier)."""
        return int(lib().pa_pool_block_bytes(self.handle))

    def swap_blocks(self, host_buffer, blocks, slots, direction, stream=None):
        """Copy whole blocks between the pool and `host_buffer` (a uint8 CPU
        tensor of whole slots, pinned for asynchronous copies): direction
        "out" copies blocks[i] -> slot slots[i], "in" slot slots[i] -> blocks[i]."""
        b_ = np.ascontiguousarray(blocks, dtype=np.int32)
        s_ = np.ascontiguousarray(slots, dtype=np.int32)
        assert b_.size == s_.size and host_buffer.dtype == torch.uint8 and not host_buffer.is_cuda
        assert host_buffer.is_contiguous()
        d = {"out": PA_SWAP_OUT, "in": PA_SWAP_IN}[direction]
        st = stream if stream is not None else torch.cuda.current_stream(self.device).cuda_stream
        _check(lib().pa_swap_blocks(self.handle, ctypes.c_void_p(host_buffer.data_ptr()),
                                    int(host_buffer.numel() // self.block_bytes()),
                                    b_.ctypes.data_as(ctypes.c_void_p), s_.ctypes.data_as(ctypes.c_void_p),
                                    int(b_.size), d, ctypes.c_void_p(st)))

    def append_kv(self, k_new, v_new, cu_new, ctx_lens, block_table, max_new_per_seq=0, stream=None):
        B = int(ctx_lens.shape[0])
        pa_append_kv(self.handle, k_new, v_new, cu_new, ctx_lens, block_table, B,
                     int(block_table.shape[1]) if B else 0, max_new_per_seq, stream)

    def set_decode_path(self, path, fused_combine=False, early_plan=False):
        """'auto', 'cuda_core' or 'tensor_core'; split sequences are merged by
        the separate combine kernel, or inside the decode kernel with
        fused_combine; early_plan overlaps the decode's planning with the
        preceding kernel (see pa_pool_set_decode_path)."""
        code = DECODE_PATHS[path] if isinstance(path, str) else int(path)
        code |= PA_DECODE_FUSED_COMBINE if fused_combine else 0
        code |= PA_DECODE_EARLY_PLAN if early_plan else 0
        pa_pool_set_decode_path(self.handle, code)

    def set_unit_cost(self, unit_cost_pages=-1):
        """Phantom pages per (sequence, kv head) unit in the decode's
        cost-balanced partition (see pa_pool_set_unit_cost); -1 = default."""
        pa_pool_set_unit_cost(self.handle, unit_cost_pages)

    def workspace_bytes(self, batch, num_q_heads, num_splits=0):
        return pa_decode_workspace_bytes(self.handle, batch, num_q_heads, num_splits)

    def num_splits(self, num_splits=0):
        return pa_decode_num_splits(self.handle, num_splits)

    def workspace(self, batch, num_q_heads, num_splits=0):
        n = self.workspace_bytes(batch, num_q_heads, num_splits)
        if self._ws is None or self._ws.numel() < n:
            # zeroed once: part of it holds call-tagged merge tickets
            self._ws = torch.zeros(max(n, 256), dtype=torch.uint8, device=self.device)
        return self._ws

    def decode(self, q, block_table, seq_lens, softmax_scale, out=None, workspace=None, num_splits=0,
               stream=None):
        B, Hq, D = q.shape
        if out is None:
            out = torch.empty((B, Hq, D), dtype=torch.float32, device=self.device)
        if workspace is None:
            workspace = self.workspace(B, Hq, num_splits)
        pa_decode(self.handle, q, block_table, seq_lens, B, Hq, int(block_table.shape[1]),
                  softmax_scale, out, workspace, workspace.numel(), num_splits, stream)
        return out

    def decode_step(self, k_new, v_new, q, block_table, seq_lens, softmax_scale, out=None, workspace=None,
                    num_splits=0, stream=None):
        """The decode step in one launch: store each sequence's new token
        (k_new / v_new [B, Hkv, D] bf16 bits, position seq_lens[b] - 1) and
        attend, as append_kv of one token per sequence then decode."""
        B, Hq, D = q.shape
        if out is None:
            out = torch.empty((B, Hq, D), dtype=torch.float32, device=self.device)
        if workspace is None:
            workspace = self.workspace(B, Hq, num_splits)
        _check(lib().pa_decode_step(self.handle, _ptr(k_new), _ptr(v_new), _ptr(q), _ptr(block_table),
                                    _ptr(seq_lens), int(B), int(Hq), int(block_table.shape[1]),
                                    float(softmax_scale), _ptr(out), _ptr(workspace), int(workspace.numel()),
                                    int(num_splits), _stream(stream)))
        return out

    def decode_multi(self, q, block_table, seq_lens, softmax_scale, out=None, num_splits=0, stream=None):
        """Several query tokens per sequence: q [B, n_q, Hq, D] (bf16 bits);
        query token i of sequence b sees seq_lens[b] - (n_q - 1 - i) tokens."""
        B, n_q, Hq, D = q.shape
        if out is None:
            out = torch.empty((B, n_q, Hq, D), dtype=torch.float32, device=self.device)
        n = int(lib().pa_decode_multi_workspace_bytes(self.handle, B, n_q, Hq, int(num_splits)))
        if B and n == 0:
            raise PagedAttnError(1, "pa_decode_multi_workspace_bytes refused the shape")
        if self._ws is None or self._ws.numel() < n:
            self._ws = torch.zeros(max(n, 256), dtype=torch.uint8, device=self.device)
        ws = self._ws
        _check(lib().pa_decode_multi(self.handle, _ptr(q), _ptr(block_table), _ptr(seq_lens), int(B), int(n_q),
                                     int(Hq), int(block_table.shape[1]), float(softmax_scale), _ptr(out),
                                     _ptr(ws), int(ws.numel()), int(num_splits), _stream(stream)))
        return out

    def device_error(self, stream=None):
        return pa_get_device_error(self.handle, stream)


class BlockManager:
    """Host block manager of a pool's physical blocks (see pa_bm_create): free
    list, per-sequence block tables, shared blocks with reference counts, a
    prefix cache of full blocks keyed by their token-id chain, fork and
    copy-on-write. Host memory only."""

    def __init__(self, num_blocks, block_size, prefix_cache=True):
        h = ctypes.c_void_p()
        _check(lib().pa_bm_create(int(num_blocks), int(block_size), 1 if prefix_cache else 0, ctypes.byref(h)))
        self.handle = h
        self.block_size = int(block_size)

    @staticmethod
    def _tokens(tokens):
        if tokens is None:
            return None, 0
        a = np.ascontiguousarray(tokens, dtype=np.int32)
        return a, int(a.size)

    def add_sequence(self, seq_id, tokens=None, n_tokens=None):
        """Admit a sequence; returns how many leading tokens sit in cached blocks."""
        a, n = self._tokens(tokens)
        if a is None:
            n = int(n_tokens)
        cached = ctypes.c_int32(0)
        _check(lib().pa_bm_add_sequence(self.handle, int(seq_id), None if a is None else a.ctypes.data_as(ctypes.c_void_p),
                                        n, ctypes.byref(cached)))
        return int(cached.value)

    def fork(self, parent_id, child_id):
        _check(lib().pa_bm_fork(self.handle, int(parent_id), int(child_id)))

    def append_tokens(self, seq_id, tokens=None, n_tokens=None):
        """Reserve slots for more tokens; returns the (src, dst) block copies the
        caller must do before writing (copy-on-write), at most one."""
        a, n = self._tokens(tokens)
        if a is None:
            n = int(n_tokens)
        src, dst, nc = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32(0)
        _check(lib().pa_bm_append_tokens(self.handle, int(seq_id), None if a is None else a.ctypes.data_as(ctypes.c_void_p),
                                         n, ctypes.byref(src), ctypes.byref(dst), 1, ctypes.byref(nc)))
        return [(int(src.value), int(dst.value))] if nc.value else []

    def free_sequence(self, seq_id):
        _check(lib().pa_bm_free_sequence(self.handle, int(seq_id)))

    def block_table(self, seq_id, max_blocks=None):
        """(block ids as an int32 array of length max_blocks (-1 padded) or of
        the sequence's block count, token count)."""
        nb, ln = ctypes.c_int32(0), ctypes.c_int64(0)
        if max_blocks is None:  # ask for the count first (a zero-size table)
            st = lib().pa_bm_block_table(self.handle, int(seq_id), None, 0, ctypes.byref(nb), ctypes.byref(ln))
            if st != 0 and nb.value == 0:
                _check(st)
        m = nb.value if max_blocks is None else int(max_blocks)
        t = np.full(max(m, 1), -1, dtype=np.int32)
        _check(lib().pa_bm_block_table(self.handle, int(seq_id), t.ctypes.data_as(ctypes.c_void_p), m,
                                       ctypes.byref(nb), ctypes.byref(ln)))
        return t[:m], int(ln.value)

    def num_free_blocks(self):
        return int(lib().pa_bm_num_free_blocks(self.handle))

    # ---- CPU swap tier
    def set_cpu_blocks(self, num_cpu_blocks):
        _check(lib().pa_bm_set_cpu_blocks(self.handle, int(num_cpu_blocks)))

    def num_free_cpu_blocks(self):
        return int(lib().pa_bm_num_free_cpu_blocks(self.handle))

    def swap_out(self, seq_id):
        """Move a resident sequence to host slots; returns the (gpu block,
        host slot) copies to make (PagedKVPool.swap_blocks, "out")."""
        n = len(self.block_table(seq_id)[0])
        src, dst, nc = np.zeros(max(n, 1), np.int32), np.zeros(max(n, 1), np.int32), ctypes.c_int32(0)
        _check(lib().pa_bm_swap_out(self.handle, int(seq_id), src.ctypes.data_as(ctypes.c_void_p),
                                    dst.ctypes.data_as(ctypes.c_void_p), n, ctypes.byref(nc)))
        return [(int(a), int(b)) for a, b in zip(src[:nc.value], dst[:nc.value])]

    def swap_in(self, seq_id):
        """Bring a swapped-out sequence back into fresh GPU blocks; returns the
        (host slot, gpu block) copies to make (PagedKVPool.swap_blocks, "in")."""
        n = len(self.swapped_slots(seq_id))
        src, dst, nc = np.zeros(max(n, 1), np.int32), np.zeros(max(n, 1), np.int32), ctypes.c_int32(0)
        _check(lib().pa_bm_swap_in(self.handle, int(seq_id), src.ctypes.data_as(ctypes.c_void_p),
                                   dst.ctypes.data_as(ctypes.c_void_p), n, ctypes.byref(nc)))
        return [(int(a), int(b)) for a, b in zip(src[:nc.value], dst[:nc.value])]

    def swapped_slots(self, seq_id):
        """Host slots of a swapped-out sequence, in token order."""
        n = ctypes.c_int32(0)
        st = lib().pa_bm_swapped_slots(self.handle, int(seq_id), None, 0, ctypes.byref(n))
        if st != 0 and n.value == 0:
            _check(st)
        a = np.zeros(max(n.value, 1), np.int32)
        _check(lib().pa_bm_swapped_slots(self.handle, int(seq_id), a.ctypes.data_as(ctypes.c_void_p), n.value,
                                         ctypes.byref(n)))
        return [int(x) for x in a[:n.value]]

    def ref_count(self, block):
        return int(lib().pa_bm_ref_count(self.handle, int(block)))

    def close(self):
        if self.handle:
            lib().pa_bm_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
