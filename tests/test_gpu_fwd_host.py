"""ring_attn_fwd_host (the forward from and to host memory, with the copies
overlapped over head groups) against ring_attn_fwd on the same inputs: every
output element identical, since each group is one ring_attn_fwd over its
heads and the heads are independent problems.  Also the float64 oracle on
one case, and consecutive calls with new inputs (the device buffers are
reused)."""
import numpy as np
import pytest
import torch

import ring_sequence_parallelism_gb300 as ra
from ring_sequence_parallelism_gb300.inputs import make_qkv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from ring_sequence_parallelism_gb300 import build

    build.build()
    ra._lib.load()


CASES = [
    # (B, H, Hkv, N, d, P, causal, layout, window, segments)
    (1, 8, 8, 4096, 128, 4, True, "striped", 0, None),  # groups of 1, 1, 2, 2, 1, 1 heads
    (1, 16, 16, 1024, 64, 4, True, "striped", 0, None),  # 1, 1, 3, 3, 3, 3, 1, 1
    (1, 9, 9, 1024, 128, 4, True, "contiguous", 0, None),  # 1, 1, 3, 2, 1, 1: a size on one lane only
    (1, 8, 2, 2048, 128, 4, True, "contiguous", 0, None),  # grouped K/V heads: 2 groups of 4 query heads
    (2, 1, 1, 1024, 64, 4, False, "contiguous", 0, None),  # groups across the batch
    (1, 3, 3, 1024, 128, 4, True, "striped", 0, None),  # 3 heads: one group
    (1, 4, 4, 2048, 128, 4, True, "zigzag", 0, None),
    (1, 4, 4, 2048, 128, 4, True, "striped", 300, [0, 700, 1500, 2048]),  # window and documents
]


def case_id(c):
    return f"{c[7]}-B{c[0]}-H{c[1]}/{c[2]}-N{c[3]}-d{c[4]}-P{c[5]}-w{c[8]}-s{0 if c[9] is None else len(c[9]) - 1}"


def handle(c):
    B, H, Hkv, N, d, P, causal, layout, window, segments = c
    att = ra.RingAttention(B, H, N, d, P, causal=causal, layout=layout, kv_heads=Hkv)
    if window:
        att.set_option(ra.RING_OPT_WINDOW, window)
    if segments is not None:
        att.set_segments(segments)
    return att


@pytest.mark.parametrize("case", CASES, ids=case_id)
def test_fwd_host_equals_fwd(case):
    B, H, Hkv, N, d, P = case[:6]
    q, k, v = make_qkv(B, H, N, d, seed=700 + N + H, Hkv=Hkv)
    att = handle(case)
    out_d, lse_d = att.fwd(q.cuda(), k.cuda(), v.cuda())
    att.check()
    out_d, lse_d = out_d.cpu(), lse_d.cpu()
    qh, kh, vh = (x.pin_memory() for x in (q, k, v))
    for rep in range(2):  # a second call reuses the device buffers
        out_h, lse_h = att.fwd_host(qh, kh, vh)
        torch.cuda.current_stream().synchronize()
        att.check()
        assert torch.equal(out_h, out_d) and torch.equal(lse_h, lse_d), f"call {rep}: host path differs"
    att.close()


def test_fwd_host_new_inputs_and_oracle(orc):
    """Two calls with different inputs on one handle: each result is the
    oracle's for its own inputs (no stale buffer survives between calls)."""
    B, H, N, d, P = 1, 4, 1024, 128, 4
    att = ra.RingAttention(B, H, N, d, P, causal=True, layout="striped")
    for seed in (711, 712):
        q, k, v = make_qkv(B, H, N, d, seed=seed)
        out_h, lse_h = att.fwd_host(*(x.pin_memory() for x in (q, k, v)))
        torch.cuda.current_stream().synchronize()
        att.check()
        ref_o, ref_l = orc.dense(q.reshape(B * H, N, d), k.reshape(B * H, N, d), v.reshape(B * H, N, d), True)
        d_out = float(np.abs(out_h.double().numpy().reshape(B * H, N, d) - ref_o).max())
        d_lse = float(np.abs(lse_h.double().numpy().reshape(B * H, N) - ref_l).max())
        print(f"fwd_host seed {seed}: max|dout|={d_out:.3e} max|dlse|={d_lse:.3e}")
        assert d_out <= 1e-2 and d_lse <= 1e-3
    att.close()


def test_fwd_host_options_change():
    """Options set between calls reach every group handle: a window, then
    documents, then neither, each call equal to ring_attn_fwd's result under
    the same options (16 heads: groups of two sizes on both lanes)."""
    B, H, N, d, P = 1, 16, 1024, 64, 4
    q, k, v = make_qkv(B, H, N, d, seed=720)
    qh, kh, vh = (x.pin_memory() for x in (q, k, v))
    qc, kc, vc = (x.cuda() for x in (q, k, v))
    att = ra.RingAttention(B, H, N, d, P, causal=True, layout="striped")
    ref = ra.RingAttention(B, H, N, d, P, causal=True, layout="striped")
    for window, segments in ((200, None), (0, [0, 300, 1024]), (0, None)):
        for a in (att, ref):
            a.set_option(ra.RING_OPT_WINDOW, window)
            a.set_segments(segments)
        out_d, lse_d = ref.fwd(qc, kc, vc)
        out_h, lse_h = att.fwd_host(qh, kh, vh)
        torch.cuda.current_stream().synchronize()
        att.check()
        ref.check()
        assert torch.equal(out_h, out_d.cpu()) and torch.equal(lse_h, lse_d.cpu()), (window, segments)
    att.close()
    ref.close()
