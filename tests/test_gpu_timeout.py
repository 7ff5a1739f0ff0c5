"""Failure detection without a GPU fault: every wait in the kernels is
bounded and, on expiry, records PA_DEVERR_TIMEOUT in an error word that the
host reads. Here one such wait is made to run out (an mbarrier that nothing
arrives at, given up after about a millisecond); the error bit must come back
and the context must stay usable for a decode checked against the oracle."""
import ctypes

import pytest

from paged_gqa_decode_02_gb300 import binding as B
from paged_gqa_decode_02_gb300 import workloads as W
from tests import harness as H

pytestmark = pytest.mark.gpu


def test_a_wait_that_cannot_complete_reports_and_the_gpu_stays_usable():
    from paged_gqa_decode_02_gb300 import build
    build.build()
    flags = ctypes.c_uint32(0)
    assert B.lib().pa_selftest_wait_timeout(0, 2_000_000, ctypes.byref(flags)) == 0
    assert flags.value == B.DEVERR_TIMEOUT
    wl = W.tiny()
    g, o = H.load_both(wl)
    ref, st = o.decode(wl.q_bits, wl.block_table, wl.seq_lens, wl.softmax_scale)
    assert st == 0
    H.check_attention(H.gpu_decode(g, wl), ref, "decode after an expired wait")
    assert g.device_error() == (0, 0)
    g.close()


def test_stream_read_calibration_runs_and_writes_nothing():
    """pa_stream_read (the benchmark's bandwidth calibration) reads a buffer
    and leaves the sink alone unless the fold hits its constant."""
    torch = H.torch_mod()
    buf = torch.ones(1 << 20, dtype=torch.float32, device="cuda")
    sink = torch.zeros(4, dtype=torch.int32, device="cuda")
    B.pa_stream_read(buf, sink)
    torch.cuda.synchronize()
    assert int(sink[0].item()) == 0
