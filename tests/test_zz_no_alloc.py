"""pa_decode_noalloc: decode for callers that cannot allocate device memory.

Such callers (an allocator that forbids device allocations on the hot path,
memory reserved up front, or no allocator to take a workspace from) call
pa_decode_noalloc, whose split-KV scratch is a fixed array inside the library
instead of a caller workspace. This file checks, through the C ABI, that two
calls in a row give the same outputs as pa_decode with a caller workspace
(within the decode tolerance used everywhere), and that a batch too large for
the fixed scratch is refused with a clear error. It is collected last so that
a stop at the first failure has already run every other test; it also passes
on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest

from paged_gqa_decode_02_gb300 import workloads as W
from tests import harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from paged_gqa_decode_02_gb300 import build, binding
    build.build()
    L = binding.lib()
    P, I32 = ctypes.c_void_p, ctypes.c_int32
    L.pa_decode_noalloc.argtypes = [P, P, P, P, I32, I32, I32, ctypes.c_float, P, I32, P]
    L.pa_decode_noalloc.restype = I32
    return L


def _noalloc(L, pool, q, table, lens, wl, out, splits):
    torch = H.torch_mod()
    st = L.pa_decode_noalloc(pool.handle, ctypes.c_void_p(q.data_ptr()),
                             ctypes.c_void_p(table.data_ptr()), ctypes.c_void_p(lens.data_ptr()),
                             wl.batch, wl.num_q_heads, wl.max_blocks, wl.softmax_scale,
                             ctypes.c_void_p(out.data_ptr()), splits,
                             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


@pytest.mark.parametrize("dt,splits", [("bf16", 0), ("bf16", 7), ("uint8", 0), ("uint4", 3)])
def test_noalloc_matches_decode_twice(lib, dt, splits):
    torch = H.torch_mod()
    wl = W.make_case("noalloc", 90, 3, 28, 4, 128, 16, dt, [700, 33, 1500], extra_blocks=2,
                     channel_offset_sigma=0.5 if dt != "bf16" else None)
    g, o = H.load_both(wl)
    ref = H.gpu_decode(g, wl, num_splits=splits)  # pa_decode with a caller workspace
    oref, ost = o.decode(wl.q_bits, wl.block_table, wl.seq_lens, wl.softmax_scale)  # the CPU oracle
    assert ost == 0
    q, table, lens = H.dev(wl.q_bits), H.dev(wl.block_table), H.dev(wl.seq_lens)
    for call in range(2):
        out = torch.full((wl.batch, wl.num_q_heads, wl.head_dim), float("nan"), dtype=torch.float32,
                         device="cuda")
        st = _noalloc(lib, g, q, table, lens, wl, out, splits)
        assert st == 0, lib.pa_last_error()
        torch.cuda.synchronize()
        got = out.cpu().numpy().reshape(ref.shape)
        H.check_attention(got, ref.astype(np.float64), f"noalloc call {call} {dt} splits={splits}")
        H.check_attention(got, oref, f"noalloc call {call} {dt} splits={splits} against the oracle")
    assert g.device_error() == (0, 0)
    g.close()


def test_noalloc_empty_and_invalid_calls_answer_like_decode(lib):
    """An empty batch returns PA_OK and invalid arguments get pa_decode's
    error, both before the scratch is looked up (nothing launched)."""
    wl = W.make_case("noalloc_args", 92, 2, 8, 8, 128, 16, "bf16", [16, 16])
    g, _ = H.make_pools(wl)
    assert lib.pa_decode_noalloc(g.handle, None, None, None, 0, 8, 1, 0.125, None, 0, None) == 0
    assert lib.pa_decode_noalloc(g.handle, None, None, None, -1, 8, 1, 0.125, None, 0, None) == 1
    assert lib.pa_decode_noalloc(g.handle, None, None, None, 2, 7, 1, 0.125, None, 0, None) == 1
    g.close()


def test_noalloc_rejects_batches_beyond_its_scratch(lib):
    wl = W.make_case("noalloc_big", 91, 2, 8, 8, 128, 16, "bf16", [16, 16])
    g, _ = H.make_pools(wl)
    big_batch = 1 << 16  # scratch need far above 8 MiB; refused before any launch
    torch = H.torch_mod()
    buf = torch.zeros(64, dtype=torch.float32, device="cuda")  # never read: the call is refused first
    ptr = ctypes.c_void_p(buf.data_ptr())
    st = lib.pa_decode_noalloc(g.handle, ptr, ptr, ptr, big_batch, 8, 1, 0.125, ptr, 0, None)
    assert st == 3
    msg = lib.pa_last_error().decode()
    assert "static scratch holds" in msg and "8388608" in msg
    g.close()
