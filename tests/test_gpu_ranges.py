"""GPU parity over wide value ranges: large per-channel offsets of K and V
(the zero-point term then cancels most of every score and of every P.V sum),
and sharp and flat softmax temperatures, for every KV format, both decode
kernels and groups of 4 and 8 query heads. The pool must match the oracle's
bit for bit and the attention stay within the usual tolerance."""
import math

import pytest

from paged_gqa_decode_02_gb300 import workloads as W
from tests import harness as H

pytestmark = pytest.mark.gpu

SEQ = [1, 17, 200, 33, 512, 90]


def _paths(dt, head_dim):
    return ["cuda_core", "tensor_core"] if dt == "bf16" or head_dim == 128 else ["cuda_core"]


@pytest.mark.parametrize("dt", ["bf16", "uint8", "uint4", "fp8"])
@pytest.mark.parametrize("sigma", [5.0, 10.0])
@pytest.mark.parametrize("hq", [8, 16])
def test_large_channel_offsets(dt, sigma, hq):
    bs = 32 if dt == "uint4" else 16
    wl = W.make_case(f"offsets_{dt}_{sigma}_{hq}", 201 + hq, len(SEQ), hq, 2, 128, bs, dt, SEQ,
                     extra_blocks=2, channel_offset_sigma=sigma)
    g, o = H.load_both(wl)
    H.assert_pools_equal(g, o)
    ref, st = o.decode(wl.q_bits, wl.block_table, wl.seq_lens, wl.softmax_scale)
    assert st == 0
    for path in _paths(dt, wl.head_dim):
        for splits in (0, 7):
            got = H.gpu_decode(g, wl, num_splits=splits, path=path)
            H.check_attention(got, ref, f"{wl.name} {path} splits={splits}")
    assert g.device_error() == (0, 0)
    g.close()


@pytest.mark.parametrize("dt", ["bf16", "uint8", "uint4", "fp8"])
@pytest.mark.parametrize("temp", [8.0, 1.0 / 64.0])
def test_sharp_and_flat_softmax(dt, temp):
    bs = 32 if dt == "uint4" else 16
    wl = W.make_case(f"temp_{dt}_{temp}", 301, len(SEQ), 8, 2, 128, bs, dt, SEQ, extra_blocks=2,
                     channel_offset_sigma=0.5 if dt != "bf16" else None,
                     softmax_scale=temp / math.sqrt(128))
    g, o = H.load_both(wl)
    ref, st = o.decode(wl.q_bits, wl.block_table, wl.seq_lens, wl.softmax_scale)
    assert st == 0
    for path in _paths(dt, wl.head_dim):
        got = H.gpu_decode(g, wl, path=path)
        H.check_attention(got, ref, f"{wl.name} {path}")
    assert g.device_error() == (0, 0)
    g.close()
