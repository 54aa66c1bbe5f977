"""The zigzag layout (2P chunks, shard r holding chunks r and 2P-1-r) with a
causal sliding window, packed documents and short queries, on the GPU
against the float64 oracle, through the C ABI.

A shard's (or block's) positions increase with its local index, so the keys
a query may see in a block stay one local interval; the kernels take its
bounds from global positions.  Forward: every row, the three rotation modes
bit for bit, block partials, the one-launch lap.  Backward: every gradient
element.  Decode: queries at the end of the cache of a zigzag handle (the
cache is read in natural order, so the layout does not enter).  Tolerances
as in the other GPU tests."""
import numpy as np
import pytest
import torch

import oracle
import ring_sequence_parallelism_gb300 as ra
from oracle import LAYOUT_ZIGZAG
from ring_sequence_parallelism_gb300.inputs import make_dout, make_qkv

pytestmark = pytest.mark.gpu

TOL_OUT = 1e-2
TOL_LSE = 1e-3
TOL_REL_L2 = 1e-2
TOL_MAX = 1e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from ring_sequence_parallelism_gb300 import build

    build.build()
    ra._lib.load()


def handle(B, H, N, d, P, causal, window=0, bounds=None):
    att = ra.RingAttention(B, H, N, d, P, causal=causal, layout="zigzag")
    if window:
        att.set_option(ra.RING_OPT_WINDOW, window)
    if bounds is not None:
        att.set_segments(bounds)
    return att


CASES = [
    # (B, H, N, d, P, causal, window, bounds)
    (1, 2, 4 * 512, 128, 4, True, 300, None),
    (1, 2, 8 * 256, 128, 8, True, 1, None),
    (1, 2, 4 * 768, 128, 4, True, 1000, None),  # chunks of 384: tile pairs span two chunks
    (1, 2, 2 * 512, 64, 2, True, 129, None),
    (1, 2, 4 * 512, 128, 4, True, 0, [0, 100, 101, 1300, 2048]),
    (1, 2, 4 * 512, 128, 4, False, 0, [0, 700, 2048]),
    (2, 1, 4 * 256, 128, 4, True, 200, [0, 333, 1024]),
    (1, 2, 4 * 512, 128, 4, True, 0, [0, 1900, 2048]),  # a valid length of 1900
]


def case_id(c):
    return f"N{c[2]}-d{c[3]}-P{c[4]}-{'c' if c[5] else 'nc'}-w{c[6]}-s{0 if c[7] is None else len(c[7]) - 1}"


@pytest.mark.parametrize("case", CASES, ids=case_id)
def test_zigzag_fwd_masks(orc, case):
    B, H, N, d, P, causal, window, bounds = case
    q, k, v = make_qkv(B, H, N, d, seed=950 + N + window)
    BH = B * H
    flat = lambda t: t.reshape(BH, N, d)
    ref_o, ref_l = orc.dense(flat(q), flat(k), flat(v), causal, window=window, segments=bounds)
    outs = []
    for mode in (2, 1, 0):
        att = handle(B, H, N, d, P, causal, window, bounds)
        att.set_option(ra.RING_OPT_ROTATION, mode)
        out, lse = att.fwd(q.cuda(), k.cuda(), v.cuda())
        att.check()
        outs.append((out.cpu(), lse.cpu()))
        att.close()
    o = outs[0][0].double().numpy().reshape(BH, N, d)
    l = outs[0][1].double().numpy().reshape(BH, N)
    d_out, d_lse = float(np.abs(o - ref_o).max()), float(np.abs(l - ref_l).max())
    print(f"zigzag {case_id(case)}: max|dout|={d_out:.3e} max|dlse|={d_lse:.3e}")
    assert d_out <= TOL_OUT and d_lse <= TOL_LSE
    for o2, l2 in outs[1:]:
        assert torch.equal(o2, outs[0][0]) and torch.equal(l2, outs[0][1]), "rotation modes differ"
    # the lap schedule, against the oracle
    att = handle(B, H, N, d, P, causal, window, bounds)
    att.set_option(ra.RING_OPT_FWD_LAP, 1)
    out, lse = att.fwd(q.cuda(), k.cuda(), v.cuda())
    att.check()
    att.close()
    d_out = float(np.abs(out.cpu().double().numpy().reshape(BH, N, d) - ref_o).max())
    d_lse = float(np.abs(lse.cpu().double().numpy().reshape(BH, N) - ref_l).max())
    print(f"zigzag lap {case_id(case)}: max|dout|={d_out:.3e} max|dlse|={d_lse:.3e}")
    assert d_out <= TOL_OUT and d_lse <= TOL_LSE


@pytest.mark.parametrize("window,bounds", [(300, None), (0, [0, 77, 300, 301, 900, 1024])])
def test_zigzag_block_partial_masks(orc, window, bounds):
    """Block partials (shard-major inputs) with a window or documents against
    the oracle's block states, every (shard, step)."""
    B, H, n, d, P = 1, 2, 256, 128, 4
    N = n * P
    q, k, v = make_qkv(B, H, N, d, seed=961)
    att = handle(B, H, N, d, P, True, window, bounds)
    pos = np.array([[orc.position(LAYOUT_ZIGZAG, n, P, r, i) for i in range(n)] for r in range(P)])
    worst_o = worst_l = 0.0
    for r in range(P):
        for s in range(P):
            j = orc.block_at(P, r, s)
            q_sh = q[:, :, pos[r]].contiguous()
            k_bl, v_bl = k[:, :, pos[j]].contiguous(), v[:, :, pos[j]].contiguous()
            st = att.new_state()
            att.block_partial(r, s, q_sh.cuda(), k_bl.cuda(), v_bl.cuda(), st, 0)
            att.check()
            m, l_, o = (x.cpu().double().numpy().reshape(B * H, n, *x.shape[3:]) for x in st)
            rm, rl, ro = orc.block_partial(q_sh.reshape(B * H, n, d), k_bl.reshape(B * H, n, d),
                                           v_bl.reshape(B * H, n, d), P, True, LAYOUT_ZIGZAG, r, j, window=window,
                                           segments=bounds)
            live = rl > 0
            assert np.array_equal(l_ > 0, live), (r, s)
            if live.any():
                worst_o = max(worst_o, float(np.abs(o[live] / l_[live][:, None] - ro[live] / rl[live][:, None]).max()))
                worst_l = max(worst_l, float(np.abs((m[live] + np.log(l_[live])) - (rm[live] + np.log(rl[live]))).max()))
    print(f"zigzag block partial w={window} s={bounds}: max|dout|={worst_o:.3e} max|dlse|={worst_l:.3e}")
    assert worst_o <= TOL_OUT and worst_l <= TOL_LSE
    att.close()


BWD_CASES = [
    (1, 2, 4 * 512, 128, 4, True, 300, None),
    (1, 2, 4 * 768, 128, 4, True, 1000, None),
    (1, 2, 4 * 512, 128, 4, True, 0, [0, 100, 101, 1300, 2048]),
    (1, 2, 4 * 512, 64, 4, False, 0, [0, 700, 2048]),
    (2, 1, 4 * 256, 128, 4, True, 200, [0, 333, 1024]),
]


@pytest.mark.parametrize("case", BWD_CASES, ids=case_id)
@pytest.mark.parametrize("lap", [True, False])
def test_zigzag_bwd_masks(orc, case, lap):
    B, H, N, d, P, causal, window, bounds = case
    q, k, v = make_qkv(B, H, N, d, seed=970 + N + window)
    do = make_dout(B, H, N, d, seed=970 + N + window)
    att = handle(B, H, N, d, P, causal, window, bounds)
    att.set_option(ra.RING_OPT_BWD_LAP, 1 if lap else 0)
    qc, kc, vc, doc = (x.cuda() for x in (q, k, v, do))
    out, lse = att.fwd(qc, kc, vc)
    got = att.bwd(qc, kc, vc, out, lse, doc)
    att.check()
    att.close()
    BH = B * H
    flat = lambda t: t.reshape(BH, N, d)
    ref = orc.dense_bwd(flat(q), flat(k), flat(v), flat(do), causal, window=window, segments=bounds)
    msg = []
    for name, a, b in zip(("dq", "dk", "dv"), got, ref):
        a = flat(a.cpu()).double().numpy()
        err = np.abs(a - b)
        rel2 = float(np.linalg.norm(a - b) / np.linalg.norm(b))
        rmax = float(err.max() / np.abs(b).max())
        msg.append(f"{name}: rel L2 {rel2:.2e}, max {rmax:.2e} of max|ref|")
        assert rel2 <= TOL_REL_L2 and rmax <= TOL_MAX, (name, rel2, rmax)
    print(f"zigzag bwd {case_id(case)} lap={lap}: " + "; ".join(msg))


@pytest.mark.parametrize("Lq,window,bounds", [(1, 0, None), (5, 0, None), (130, 0, None), (300, 0, None),
                                               (64, 500, None), (200, 0, [0, 1000, 1900, 4096])])
def test_zigzag_decode(orc, Lq, window, bounds):
    """Short queries at positions N-Lq .. N-1 over the cache of a zigzag
    handle with a window or documents, against the oracle's dense rows."""
    B, H, N, d, P = 1, 4, 4096, 128, 4
    q_all, k, v = make_qkv(B, H, N, d, seed=980 + Lq)
    q = q_all[:, :, N - Lq:].contiguous()
    att = handle(B, H, N, d, P, True, window, bounds)
    out, lse = att.decode(q.cuda(), k.cuda(), v.cuda())
    att.check()
    att.close()
    BH = B * H
    rows = np.arange(N - Lq, N)
    ref_o, ref_l = orc.dense(q_all.reshape(BH, N, d), k.reshape(BH, N, d), v.reshape(BH, N, d), True, rows=rows,
                             window=window, segments=bounds)
    d_out = float(np.abs(out.cpu().double().numpy().reshape(BH, Lq, d) - ref_o).max())
    d_lse = float(np.abs(lse.cpu().double().numpy().reshape(BH, Lq) - ref_l).max())
    print(f"zigzag decode Lq={Lq} w={window} s={bounds}: max|dout|={d_out:.3e} max|dlse|={d_lse:.3e}")
    assert d_out <= TOL_OUT and d_lse <= TOL_LSE
