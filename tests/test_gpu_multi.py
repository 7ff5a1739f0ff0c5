"""GPU parity of the decode with several query tokens per sequence
(pa_decode_multi: chunked prefill, speculative verification) against the
oracle's causal attention: query token i of n_q sees the first
seq_len - (n_q - 1 - i) tokens. Covers every KV format, group sizes that
give one to eight query tokens per column group, sequences shorter than the
chunk (zero rows), split counts from one to many slices per sequence, both
decode kernels and the early-plan launch."""
import numpy as np
import pytest

from paged_gqa_decode_02_gb300 import workloads as W
from tests import harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_gqa_decode_02_gb300 import build
    build.build()


def _paths(dt, head_dim):
    return ["cuda_core", "tensor_core"] if dt == "bf16" or head_dim == 128 else ["cuda_core"]


def _run(g, wl, q, path, splits, early):
    """Decode into an output with guard regions on both sides (canaries: no
    row may be written outside the [B, n_q, Hq, D] output)."""
    torch = H.torch_mod()
    g.set_decode_path(path, early_plan=early)
    n, GO = int(np.prod(q.shape)), 1024
    obuf = torch.full((n + 2 * GO,), 12345.0, dtype=torch.float32, device="cuda")
    out = obuf[GO:GO + n].view(*q.shape)
    out.fill_(float("nan"))
    g.decode_multi(H.dev(q), H.dev(wl.block_table), H.dev(wl.seq_lens), wl.softmax_scale, out=out,
                   num_splits=splits)
    torch.cuda.synchronize()
    assert bool((obuf[:GO] == 12345.0).all()) and bool((obuf[GO + n:] == 12345.0).all()), "output guard"
    return out.cpu().numpy().reshape(-1, wl.head_dim)


@pytest.mark.parametrize("dt", ["bf16", "uint8", "uint4", "fp8"])
@pytest.mark.parametrize("g_heads,n_q", [(7, 2), (4, 3), (2, 5), (1, 8), (4, 8)])
def test_multi_token_queries(dt, g_heads, n_q):
    seq = [3 * n_q, 1, n_q - 1, 200, 17, 0, 65]
    D = 128 if dt in ("uint4", "fp8") or g_heads != 2 else 64
    wl = W.make_case(f"mq_{dt}_{g_heads}_{n_q}", 61 + n_q, len(seq), 2 * g_heads, 2, D, 16, dt, seq,
                     extra_blocks=2, channel_offset_sigma=None if dt == "bf16" else 0.5)
    gp, o = H.load_both(wl, leave_last=False)
    q = W.multi_token_queries(61 + n_q, wl.batch, n_q, wl.num_q_heads, D)
    ref, st = o.decode_multi(q, wl.block_table, wl.seq_lens, wl.softmax_scale)
    assert st == 0
    for path in _paths(dt, D):
        for splits, early in ((0, True), (1, False), (7, False), (300, True)):
            got = _run(gp, wl, q, path, splits, early)
            H.check_attention(got, ref, f"{wl.name} {path} splits={splits} early={early}")
    assert gp.device_error() == (0, 0)
    gp.close()


def test_one_query_token_is_the_decode_step():
    torch = H.torch_mod()
    wl = W.random_small(3, "bf16")
    gp, o = H.load_both(wl)
    a = H.gpu_decode(gp, wl)
    b = _run(gp, wl, wl.q_bits[:, None], "auto", 0, False)
    np.testing.assert_array_equal(np.asarray(a).reshape(-1, wl.head_dim), b)
    gp.close()
