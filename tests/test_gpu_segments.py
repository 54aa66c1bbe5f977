"""Sequence packing (ring_attn_set_segments) on the GPU against the float64
oracle: forward, block partials, the three rotation modes, short-query
decode and the backward, through the C ABI.

Tolerances as in the other GPU tests: max|d out| <= 1e-2, max|d lse| <= 1e-3
(bf16 inputs, fp32 accumulation); gradients: relative L2 <= 1e-2 and max
error <= 2e-2 of the largest magnitude (see tests/test_gpu_backward.py for
the derivation)."""
import numpy as np
import pytest
import torch

import oracle
import ring_sequence_parallelism_gb300 as ra
from ring_sequence_parallelism_gb300.inputs import WORKLOADS, document_bounds, make_dout, make_qkv, make_workload, \
    sample_rows

pytestmark = pytest.mark.gpu

TOL_OUT = 1e-2
TOL_LSE = 1e-3


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from ring_sequence_parallelism_gb300 import build

    build.build()
    ra._lib.load()


def handle(B, H, N, d, P, causal, layout, bounds, window=0):
    att = ra.RingAttention(B, H, N, d, P, causal=causal, layout=layout)
    if window:
        att.set_option(ra.RING_OPT_WINDOW, window)
    att.set_segments(bounds)
    return att


CASES = [
    # (B, H, N, d, P, causal, layout, window, bounds)
    (1, 2, 1024, 128, 4, True, "striped", 0, [0, 100, 101, 613, 1024]),
    (1, 2, 1024, 128, 4, True, "contiguous", 0, [0, 100, 101, 613, 1024]),
    (1, 2, 1024, 64, 4, False, "contiguous", 0, [0, 300, 1000, 1024]),  # non-causal: block diagonal
    (1, 2, 1024, 128, 4, False, "striped", 0, [0, 300, 1000, 1024]),
    (1, 2, 3 * 328, 128, 3, True, "contiguous", 0, [0, 129, 500, 984]),  # ragged shards
    (1, 2, 3 * 328, 128, 3, True, "striped", 0, [0, 129, 500, 984]),
    (2, 1, 2048, 128, 8, True, "striped", 200, [0, 700, 1500, 2048]),  # with a sliding window
    (1, 2, 2048, 128, 4, True, "contiguous", 333, [0, 1, 2, 1030, 2048]),
    (1, 2, 2048, 128, 4, True, "striped", 0, [0, 1900, 2048]),  # a valid length of 1900: padding
    # a document starting late in a shard: the second query tile of a CTA
    # needs key tiles that start six tiles after the first tile's
    (1, 2, 4096, 128, 4, True, "contiguous", 0, [0, 1000, 3950, 4096]),
    (1, 2, 4096, 128, 4, True, "striped", 0, [0, 1000, 3950, 4096]),
    # non-causal: in block 1 of shard 0 the first query tile has no key and
    # the second has all of them
    (1, 2, 1024, 128, 4, False, "contiguous", 0, [0, 128, 1024]),
]


def case_id(c):
    return f"{c[6]}-N{c[2]}-d{c[3]}-P{c[4]}-{'c' if c[5] else 'nc'}-w{c[7]}-s{len(c[8]) - 1}"


@pytest.mark.parametrize("case", CASES, ids=case_id)
def test_fwd_segments(orc, case):
    """Every row against the oracle's dense attention with the same
    documents; the three rotation modes give identical bits."""
    B, H, N, d, P, causal, layout, window, bounds = case
    q, k, v = make_qkv(B, H, N, d, seed=600 + N)
    BH = B * H
    ref_o, ref_l = orc.dense(q.reshape(BH, N, d), k.reshape(BH, N, d), v.reshape(BH, N, d), causal,
                             window=window, segments=bounds)
    outs = []
    for mode in (2, 1, 0):
        att = handle(B, H, N, d, P, causal, layout, bounds, window)
        att.set_option(ra.RING_OPT_ROTATION, mode)
        out, lse = att.fwd(q.cuda(), k.cuda(), v.cuda())
        att.check()
        outs.append((out.cpu(), lse.cpu()))
        att.close()
    o = outs[0][0].double().numpy().reshape(BH, N, d)
    l = outs[0][1].double().numpy().reshape(BH, N)
    d_out, d_lse = float(np.abs(o - ref_o).max()), float(np.abs(l - ref_l).max())
    print(f"segments {case_id(case)}: max|dout|={d_out:.3e} max|dlse|={d_lse:.3e}")
    assert d_out <= TOL_OUT and d_lse <= TOL_LSE
    for o2, l2 in outs[1:]:
        assert torch.equal(o2, outs[0][0]) and torch.equal(l2, outs[0][1]), "rotation modes differ"


@pytest.mark.parametrize("layout", ["contiguous", "striped"])
def test_block_partial_segments(orc, layout):
    """Block partials (shard-major inputs) against the oracle's block state
    with the same documents, for every (shard, step)."""
    B, H, n, d, P = 1, 2, 256, 128, 4
    N = n * P
    bounds = [0, 77, 300, 301, 900, N]
    q, k, v = make_qkv(B, H, N, d, seed=621)
    lid = {"contiguous": 0, "striped": 1}[layout]
    att = handle(B, H, N, d, P, True, layout, bounds)
    orc_ = oracle.default()
    pos = np.array([[orc_.position(lid, n, P, r, i) for i in range(n)] for r in range(P)])
    worst = 0.0
    for r in range(P):
        for s in range(P):
            j = orc_.block_at(P, r, s)
            q_sh = q[:, :, pos[r]].contiguous()
            k_bl, v_bl = k[:, :, pos[j]].contiguous(), v[:, :, pos[j]].contiguous()
            st = att.new_state()
            att.block_partial(r, s, q_sh.cuda(), k_bl.cuda(), v_bl.cuda(), st, 0)
            att.check()
            m, l_, o = (x.cpu().double().numpy().reshape(B * H, n, *x.shape[3:]) for x in st)
            rm, rl, ro = orc_.block_partial(q_sh.reshape(B * H, n, d), k_bl.reshape(B * H, n, d),
                                            v_bl.reshape(B * H, n, d), P, True, lid, r, j, segments=bounds)
            live = rl > 0
            if live.any():
                # compare normalised per-block outputs and log-sum-exps where a row has keys
                got_o = o[live] / l_[live][:, None]
                ref_o = ro[live] / rl[live][:, None]
                worst = max(worst, float(np.abs(got_o - ref_o).max()))
                assert np.abs((m[live] + np.log(l_[live])) - (rm[live] + np.log(rl[live]))).max() <= TOL_LSE
            assert np.all(l_[~live] == 0.0), "rows without keys must stay empty"
    print(f"block partial segments {layout}: max|dout|={worst:.3e}")
    assert worst <= TOL_OUT
    att.close()


@pytest.mark.parametrize("layout", ["contiguous", "striped"])
def test_decode_segments(orc, layout):
    """Short queries at the end of a packed sequence see only their own
    document's cached keys."""
    B, H, N, d, P, Lq = 1, 2, 4096, 128, 4, 200
    bounds = [0, 1000, 3950, N]  # the last document starts inside the query block
    q_all, k, v = make_qkv(B, H, N, d, seed=631)
    q = q_all[:, :, N - Lq:].contiguous()
    att = handle(B, H, N, d, P, True, layout, bounds)
    out, lse = att.decode(q.cuda(), k.cuda(), v.cuda())
    att.check()
    BH = B * H
    rows = np.arange(N - Lq, N)
    ref_o, ref_l = orc.dense(q_all.reshape(BH, N, d), k.reshape(BH, N, d), v.reshape(BH, N, d), True, rows=rows,
                             segments=bounds)
    d_out = float(np.abs(out.cpu().double().numpy().reshape(BH, Lq, d) - ref_o).max())
    d_lse = float(np.abs(lse.cpu().double().numpy().reshape(BH, Lq) - ref_l).max())
    print(f"decode segments {layout}: max|dout|={d_out:.3e} max|dlse|={d_lse:.3e}")
    assert d_out <= TOL_OUT and d_lse <= TOL_LSE
    att.close()


BWD_CASES = [
    (1, 2, 1024, 128, 4, True, "striped", 0, [0, 100, 101, 613, 1024]),
    (1, 2, 1024, 128, 4, True, "contiguous", 0, [0, 100, 101, 613, 1024]),
    (1, 2, 1024, 64, 4, False, "striped", 0, [0, 300, 1000, 1024]),
    (1, 2, 3 * 328, 128, 3, True, "contiguous", 150, [0, 129, 500, 984]),
]


@pytest.mark.parametrize("case", BWD_CASES, ids=case_id)
def test_bwd_segments(orc, case):
    from test_gpu_backward import check_grads

    B, H, N, d, P, causal, layout, window, bounds = case
    q, k, v = make_qkv(B, H, N, d, seed=640 + N)
    do = make_dout(B, H, N, d, seed=640 + N)
    att = handle(B, H, N, d, P, causal, layout, bounds, window)
    qc, kc, vc, doc = (x.cuda() for x in (q, k, v, do))
    out, lse = att.fwd(qc, kc, vc)
    dq, dk, dv = att.bwd(qc, kc, vc, out, lse, doc)
    att.check()
    BH = B * H
    flat = lambda t: t.reshape(BH, N, d)
    ref = orc.dense_bwd(flat(q), flat(k), flat(v), flat(do), causal, window=window, segments=bounds)
    check_grads(f"bwd segments {case_id(case)}", [flat(g).cpu().numpy() for g in (dq, dk, dv)], ref)
    att.close()


def test_fwd_packed_128k_sampled(orc):
    """The 128K striped workload packed with documents of 1K-16K tokens:
    256 sampled rows per head (plus each document's first and last row)
    against the oracle."""
    w = WORKLOADS["packed-128k"]
    bounds = w.segments()
    q, k, v = make_workload(w)
    att = handle(w.B, w.H, w.N, w.d, w.P, w.causal, w.layout, bounds)
    out, lse = att.fwd(q.cuda(), k.cuda(), v.cuda())
    att.check()
    extra = tuple(bounds[:-1]) + tuple(b - 1 for b in bounds[1:])
    rows = sample_rows(w.N, 256, extra=extra).numpy()
    BH = w.B * w.H
    ref_o, ref_l = orc.dense(q.reshape(BH, w.N, w.d), k.reshape(BH, w.N, w.d), v.reshape(BH, w.N, w.d), True,
                             rows=rows, segments=bounds)
    o = out.reshape(BH, w.N, w.d)[:, rows].cpu().double().numpy()
    l = lse.reshape(BH, w.N)[:, rows].cpu().double().numpy()
    d_out, d_lse = float(np.abs(o - ref_o).max()), float(np.abs(l - ref_l).max())
    print(f"packed-128k sampled: max|dout|={d_out:.3e} max|dlse|={d_lse:.3e}")
    assert d_out <= TOL_OUT and d_lse <= TOL_LSE
    att.close()
