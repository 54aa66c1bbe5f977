"""CUDA path against the float64 oracle, element by element (GPU only).

Tolerances (bf16 inputs, fp32 accumulation): max|d out| <= 1e-2 and
max|d lse| <= 1e-3; the fp32 merge of fp32 states: <= 1e-5.  Every call goes
through the C ABI (the ctypes binding)."""
import numpy as np
import pytest
import torch

import oracle
import ring_sequence_parallelism_gb300 as ra
from oracle import LAYOUT_CONTIGUOUS, LAYOUT_STRIPED, LAYOUT_ZIGZAG
from ring_sequence_parallelism_gb300.inputs import WORKLOADS, expand_kv, make_qkv, make_workload, sample_rows

pytestmark = pytest.mark.gpu

TOL_OUT = 1e-2
TOL_LSE = 1e-3
TOL_MERGE = 1e-5


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from ring_sequence_parallelism_gb300 import build

    build.build()
    ra._lib.load()


def lid(layout):
    return {"contiguous": LAYOUT_CONTIGUOUS, "striped": LAYOUT_STRIPED, "zigzag": LAYOUT_ZIGZAG}[layout]


def flat(t, BH):
    return t.reshape(BH, *t.shape[2:])


def report(name, out, lse, ref_out, ref_lse):
    d_out = float(np.max(np.abs(out - ref_out))) if out.size else 0.0
    d_lse = float(np.max(np.abs(lse - ref_lse))) if lse.size else 0.0
    print(f"{name}: max|dout|={d_out:.3e} max|dlse|={d_lse:.3e}")
    return d_out, d_lse


def run_fwd(B, H, N, d, P, causal, layout, q, k, v, rotation=None, window=0):
    att = ra.RingAttention(B, H, N, d, P, causal=causal, layout=layout, kv_heads=k.shape[1])
    if window:
        att.set_option(ra.RING_OPT_WINDOW, window)
    if rotation is not None:
        att.set_option(ra.RING_OPT_ROTATION, rotation)
    out, lse = att.fwd(q.cuda(), k.cuda(), v.cuda())
    att.check()
    torch.cuda.synchronize()
    res = out.cpu(), lse.cpu()
    att.close()
    return res


# ------------------------------------------------------------ merge et al.
def random_state(rows, d, seed, empty_frac=0.1):
    g = np.random.default_rng(seed)
    m = g.normal(0, 3, rows).astype(np.float32)
    l = g.uniform(0.5, 4.0, rows).astype(np.float32)
    o = g.normal(0, 1, (rows, d)).astype(np.float32)
    empty = g.random(rows) < empty_frac
    m[empty] = -np.inf
    l[empty] = 0.0
    o[empty] = 0.0
    return m, l, o


@pytest.mark.parametrize("B,H,n,d,offset", [(1, 2, 128, 64, 0), (2, 3, 200, 128, 0), (1, 8, 1024, 128, 0),
                                             (2, 3, 200, 128, 4), (1, 2, 131, 64, 4)])
def test_merge_matches_oracle(B, H, n, d, offset):
    """The fp32 merge of two fp32 states against the oracle's float64 merge
    of the same states (<= 1e-5).  offset 4 places both O~ arrays 16 bytes
    past a 32-byte boundary, so the kernel takes its 128-bit path."""
    P = 2
    att = ra.RingAttention(B, H, n * P, d, P, causal=True, layout="striped")
    rows = B * H * n
    a = random_state(rows, d, 1)
    b = random_state(rows, d, 2)
    # also rows where both sides are empty, and equal maxima
    a[0][:3] = -np.inf; a[1][:3] = 0; a[2][:3] = 0
    b[0][:2] = -np.inf; b[1][:2] = 0; b[2][:2] = 0
    b[0][5] = a[0][5]
    def to_gpu(x):
        t = torch.from_numpy(x.reshape((B, H, n) + x.shape[1:]))
        if x.ndim == 1 or not offset:
            return t.cuda().contiguous()
        buf = torch.empty(t.numel() + offset, dtype=t.dtype, device="cuda")
        g = buf[offset:].view(t.shape)
        g.copy_(t)
        assert g.data_ptr() % 32 == 16
        return g

    ga = tuple(to_gpu(x) for x in a)
    gb = tuple(to_gpu(x) for x in b)
    att.merge(ga, gb)
    torch.cuda.synchronize()
    m, l, o = (x.cpu().numpy().reshape(rows, -1).squeeze() for x in ga)
    o = ga[2].cpu().numpy().reshape(rows, d)
    rm, rl, ro = oracle.default().merge_states(a, b)
    both_empty = np.isneginf(rm)
    assert np.array_equal(np.isneginf(m), both_empty)
    assert np.all(l[both_empty] == 0) and np.all(o[both_empty] == 0)
    ne = ~both_empty
    assert np.max(np.abs(m[ne] - rm[ne])) <= TOL_MERGE
    assert np.max(np.abs(l[ne] - rl[ne])) <= TOL_MERGE * max(1.0, float(np.max(rl)))
    assert np.max(np.abs(o[ne] - ro[ne])) <= TOL_MERGE
    att.close()


def test_state_init_and_finalize():
    B, H, N, d, P = 1, 2, 4 * 200, 128, 4
    att = ra.RingAttention(B, H, N, d, P, causal=True, layout="striped")
    st = att.new_state()
    att.state_init(st)
    torch.cuda.synchronize()
    assert torch.all(torch.isneginf(st[0])) and torch.all(st[1] == 0) and torch.all(st[2] == 0)
    rows = B * H * att.n
    m, l, o = random_state(rows, d, 7)
    st = tuple(torch.from_numpy(x.reshape((B, H, att.n) + x.shape[1:])).cuda().contiguous() for x in (m, l, o))
    out = torch.full((B, H, N, d), 7.0, device="cuda")
    lse = torch.full((B, H, N), 7.0, device="cuda")
    r = 2
    att.finalize(r, st, out, lse)
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle.default().finalize(m, l, o)
    pos = [i * P + r for i in range(att.n)]
    got_out = out.cpu().numpy().reshape(B * H, N, d)[:, pos].reshape(rows, d)
    got_lse = lse.cpu().numpy().reshape(B * H, N)[:, pos].reshape(rows)
    fin = np.isfinite(ref_lse)
    assert np.max(np.abs(got_out - ref_out)) <= 1e-6
    assert np.max(np.abs(got_lse[fin] - ref_lse[fin])) <= 1e-6
    assert np.all(np.isneginf(got_lse[~fin]))
    others = [t for t in range(N) if t % P != r]
    assert torch.all(out.reshape(B * H, N, d)[:, others] == 7.0)
    att.close()


# ------------------------------------------------------------ block partial
@pytest.mark.parametrize("layout,n", [("contiguous", 128), ("contiguous", 328), ("striped", 128), ("striped", 328),
                                      ("zigzag", 256), ("zigzag", 512)])
@pytest.mark.parametrize("d", [64, 128])
def test_block_partial_matches_oracle(layout, d, n):
    """Every (shard, step) block of a small ring, fresh (accumulate 0): the
    block state's unique parts, m + ln l and O~/l, against the oracle's block
    partial; empty rows must come back as (m=-inf, l=0, O~=0)."""
    B, H, P = 1, 2, 3
    N = n * P
    q, k, v = make_qkv(B, H, N, d, seed=n + d)
    att = ra.RingAttention(B, H, N, d, P, causal=True, layout=layout)
    orc = oracle.default()
    L = lid(layout)
    BH = B * H
    qf, kf, vf = flat(q, BH), flat(k, BH), flat(v, BH)
    worst_o = worst_l = 0.0
    for r in range(P):
        pos_r = [orc.position(L, n, P, r, i) for i in range(n)]
        q_sh = qf[:, pos_r].contiguous()
        for s in range(P):
            j = orc.block_at(P, r, s)
            pos_j = [orc.position(L, n, P, j, i) for i in range(n)]
            k_bl, v_bl = kf[:, pos_j].contiguous(), vf[:, pos_j].contiguous()
            st = att.new_state()
            for x in st:
                x.fill_(float("nan"))
            att.block_partial(r, s, q_sh.reshape(B, H, n, d).cuda(), k_bl.reshape(B, H, n, d).cuda(),
                              v_bl.reshape(B, H, n, d).cuda(), st, 0)
            att.check()
            m, l, o = (x.cpu().double().numpy().reshape(BH * n, -1) for x in st)
            m, l = m[:, 0], l[:, 0]
            rm, rl, ro = orc.block_partial(q_sh, k_bl, v_bl, P, True, L, r, j)
            rm, rl, ro = rm.reshape(-1), rl.reshape(-1), ro.reshape(BH * n, d)
            empty = np.isneginf(rm)
            assert np.all(np.isneginf(m[empty])) and np.all(l[empty] == 0) and np.all(o[empty] == 0), (r, s)
            ne = ~empty
            if ne.any():
                dl = np.abs((m[ne] + np.log(l[ne])) - (rm[ne] + np.log(rl[ne])))
                do = np.abs(o[ne] / l[ne][:, None] - ro[ne] / rl[ne][:, None])
                worst_l, worst_o = max(worst_l, float(dl.max())), max(worst_o, float(do.max()))
    print(f"block partial {layout} d={d} n={n}: max|dout|={worst_o:.3e} max|dlse|={worst_l:.3e}")
    assert worst_o <= TOL_OUT and worst_l <= TOL_LSE
    att.close()


@pytest.mark.parametrize("layout", ["contiguous", "striped", "zigzag"])
def test_block_partial_ring_with_accumulate(layout):
    """The pages' loop driven through the C ABI: empty state, then P block
    partials with accumulate 1 in ring order, then finalize; equals dense
    attention (oracle)."""
    B, H, n, d, P = 1, 2, 256, 128, 4
    N = n * P
    q, k, v = make_qkv(B, H, N, d, seed=77)
    att = ra.RingAttention(B, H, N, d, P, causal=True, layout=layout)
    orc = oracle.default()
    L = lid(layout)
    BH = B * H
    qf, kf, vf = flat(q, BH), flat(k, BH), flat(v, BH)
    out = torch.empty((B, H, N, d), device="cuda")
    lse = torch.empty((B, H, N), device="cuda")
    for r in range(P):
        pos_r = [orc.position(L, n, P, r, i) for i in range(n)]
        st = att.new_state()
        att.state_init(st)
        for s in range(P):
            j = orc.block_at(P, r, s)
            pos_j = [orc.position(L, n, P, j, i) for i in range(n)]
            att.block_partial(r, s, qf[:, pos_r].reshape(B, H, n, d).cuda(), kf[:, pos_j].reshape(B, H, n, d).cuda(),
                              vf[:, pos_j].reshape(B, H, n, d).cuda(), st, 1)
        att.finalize(r, st, out, lse)
    att.check()
    ref_out, ref_lse = orc.dense(qf, kf, vf, True)
    d_out, d_lse = report(f"block ring {layout}", out.cpu().double().numpy().reshape(BH, N, d),
                          lse.cpu().double().numpy().reshape(BH, N), ref_out, ref_lse)
    assert d_out <= TOL_OUT and d_lse <= TOL_LSE
    att.close()


# ------------------------------------------------------------ ring forward
SMALL_CASES = [
    # (B, H, N, d, P, causal, layout)
    (1, 2, 512, 64, 4, False, "contiguous"),    # 2 heads x 512 tokens, non-causal
    (1, 2, 512, 64, 4, True, "striped"),
    (2, 2, 3 * 200, 128, 3, True, "contiguous"),  # ragged tail (n = 200)
    (2, 2, 3 * 200, 128, 3, True, "striped"),
    (1, 3, 640, 128, 1, True, "contiguous"),      # P = 1: one block, one step
    (1, 1, 5 * 8, 64, 5, True, "striped"),        # n = 8: tiny shards
    (1, 2, 2048, 128, 16, True, "striped"),
    (1, 2, 2048, 128, 2, False, "striped"),
    # shard lengths around the tile edges: n = 129 and 257 leave a last key
    # tile that no query of a j > r striped block uses (it is still sent);
    # n = 1 has no allowed pair at all in those blocks
    (1, 2, 4 * 129, 64, 4, True, "striped"),
    (1, 2, 3 * 257, 128, 3, True, "striped"),
    (1, 2, 4 * 1, 64, 4, True, "striped"),
    # FULL blocks walk their key tiles in rotated order; n = 328 puts the
    # ragged tile first for the CTA of query tiles 0, 1
    (1, 2, 3 * 328, 128, 3, True, "contiguous"),
    (1, 2, 2 * 328, 64, 2, False, "striped"),
    # zigzag: chunks of 128 tokens put tile 0 in the early chunk and tile 1
    # in the late one (one tile pair spans both); chunks of 256 and 512
    (1, 2, 4 * 256, 64, 4, True, "zigzag"),
    (2, 2, 3 * 512, 128, 3, True, "zigzag"),
    (1, 2, 8 * 1024, 128, 8, True, "zigzag"),
    (1, 2, 2 * 256, 128, 2, False, "zigzag"),
    (1, 3, 256, 128, 1, True, "zigzag"),
]


@pytest.mark.parametrize("case", SMALL_CASES, ids=lambda c: "B{}H{}N{}d{}P{}{}{}".format(
    c[0], c[1], c[2], c[3], c[4], "c" if c[5] else "n", c[6][0]))
def test_fwd_small(case):
    B, H, N, d, P, causal, layout = case
    q, k, v = make_qkv(B, H, N, d, seed=N + P + d)
    out, lse = run_fwd(B, H, N, d, P, causal, layout, q, k, v)
    BH = B * H
    ref_out, ref_lse = oracle.default().dense(flat(q, BH), flat(k, BH), flat(v, BH), causal)
    d_out, d_lse = report(f"fwd {case}", out.double().numpy().reshape(BH, N, d),
                          lse.double().numpy().reshape(BH, N), ref_out, ref_lse)
    assert d_out <= TOL_OUT and d_lse <= TOL_LSE


@pytest.mark.parametrize("shape", [(1, 2, 8 * 256, 128, 8), (2, 1, 5 * 200, 64, 5)])
def test_fwd_rotation_matches_direct_indexing(shape):
    """The rotation only moves bytes: sending from the step kernel (mode 2)
    and side-stream copies (mode 1) give results identical bit for bit to
    reading every block straight from the packed buffer (mode 0), for causal
    blocks of both layouts (contiguous skips blocks, whose slots the side
    stream copies in mode 2) and for non-causal FULL blocks."""
    B, H, N, d, P = shape
    q, k, v = make_qkv(B, H, N, d, seed=5)
    cases = [("contiguous", True), ("striped", True), ("contiguous", False)]
    if (N // P) % 256 == 0:
        cases.append(("zigzag", True))
    for layout, causal in cases:
        ref = run_fwd(B, H, N, d, P, causal, layout, q, k, v, rotation=0)
        for mode in (1, 2):
            got = run_fwd(B, H, N, d, P, causal, layout, q, k, v, rotation=mode)
            assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1]), (layout, causal, mode)


def test_fwd_noncausal_512_workload():
    w = WORKLOADS["noncausal-512"]
    q, k, v = make_workload(w)
    out, lse = run_fwd(w.B, w.H, w.N, w.d, w.P, w.causal, w.layout, q, k, v)
    BH = w.B * w.H
    orc = oracle.default()
    ref_out, ref_lse = orc.dense(flat(q, BH), flat(k, BH), flat(v, BH), w.causal)
    ring_out, ring_lse = orc.ring(flat(q, BH), flat(k, BH), flat(v, BH), w.P, w.causal, LAYOUT_CONTIGUOUS)
    assert np.max(np.abs(ring_out - ref_out)) <= 1e-12
    d_out, d_lse = report(w.name, out.double().numpy().reshape(BH, w.N, w.d), lse.double().numpy().reshape(BH, w.N),
                          ref_out, ref_lse)
    assert d_out <= TOL_OUT and d_lse <= TOL_LSE


def test_fwd_8k_contiguous_and_striped():
    """The 8K causal workloads in the three layouts, every row, against
    dense; then the striped and zigzag results against the contiguous one
    (same seeded inputs; outputs are in natural order, so no un-permuting is
    left to do)."""
    wc, ws, wz = WORKLOADS["contiguous-8k"], WORKLOADS["striped-8k"], WORKLOADS["zigzag-8k"]
    q, k, v = make_workload(wc)
    BH = wc.B * wc.H
    ref_out, ref_lse = oracle.default().dense(flat(q, BH), flat(k, BH), flat(v, BH), True)
    res = {}
    for w in (wc, ws, wz):
        out, lse = run_fwd(w.B, w.H, w.N, w.d, w.P, w.causal, w.layout, q, k, v)
        res[w.name] = (out, lse)
        d_out, d_lse = report(w.name, out.double().numpy().reshape(BH, w.N, w.d),
                              lse.double().numpy().reshape(BH, w.N), ref_out, ref_lse)
        assert d_out <= TOL_OUT and d_lse <= TOL_LSE
    a = res[wc.name]
    for b in (res[ws.name], res[wz.name]):
        assert float((a[0] - b[0]).abs().max()) <= 2 * TOL_OUT
        assert float((a[1] - b[1]).abs().max()) <= 2 * TOL_LSE


def _sampled_check(w, rows_per_head, ring_rows=0):
    q, k, v = make_workload(w)
    out, lse = run_fwd(w.B, w.H, w.N, w.d, w.P, w.causal, w.layout, q, k, v, window=w.window)
    k, v = expand_kv(k, w.H), expand_kv(v, w.H)  # the oracle sees each query head's K/V
    BH = w.B * w.H
    n = w.n
    # shard and chunk edges (zigzag chunks are n/2 long) and the middle
    extra = (0, 1, w.N - 1, n - 1, n, w.P - 1, w.P, w.N // 2, n // 2 - 1, n // 2, w.N - n // 2 - 1, w.N - n // 2)
    rows = sample_rows(w.N, rows_per_head, extra=extra).numpy()
    orc = oracle.default()
    qf, kf, vf = flat(q, BH), flat(k, BH), flat(v, BH)
    ref_out, ref_lse = orc.dense(qf, kf, vf, w.causal, rows=rows, window=w.window)
    got_out = out.reshape(BH, w.N, w.d)[:, rows].double().numpy()
    got_lse = lse.reshape(BH, w.N)[:, rows].double().numpy()
    d_out, d_lse = report(f"{w.name} ({rows.size} rows/head)", got_out, got_lse, ref_out, ref_lse)
    assert d_out <= TOL_OUT and d_lse <= TOL_LSE
    if ring_rows:
        rr = rows[:ring_rows]
        r_out, r_lse = orc.ring(qf, kf, vf, w.P, w.causal, w.layout_id, rows=rr, window=w.window)
        assert np.max(np.abs(r_out - ref_out[:, :ring_rows])) <= 1e-10
        assert np.max(np.abs(r_lse - ref_lse[:, :ring_rows])) <= 1e-10
    # properties that hold at any size: finite everywhere, lse above the
    # diagonal score, and causal row 0 equal to v_0
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()
    v0 = v.reshape(BH, w.N, w.d)[:, 0].float()
    assert float((out.reshape(BH, w.N, w.d)[:, 0] - v0).abs().max()) <= TOL_OUT


def test_fwd_128k_striped_sampled():
    _sampled_check(WORKLOADS["striped-128k"], 256, ring_rows=16)


def test_fwd_128k_zigzag_sampled():
    _sampled_check(WORKLOADS["zigzag-128k"], 256, ring_rows=16)


def test_fwd_128k_window_sampled():
    _sampled_check(WORKLOADS["swa-128k"], 256, ring_rows=16)


WINDOW_CASES = [
    # (B, H, N, d, P, layout, window)
    (1, 2, 4 * 256, 64, 4, "contiguous", 1),
    (1, 2, 4 * 256, 128, 4, "striped", 100),
    (2, 2, 3 * 200, 128, 3, "contiguous", 129),  # ragged shards
    (1, 2, 3 * 200, 64, 3, "striped", 300),
    (1, 2, 8 * 256, 128, 8, "striped", 700),
    (1, 2, 8 * 256, 128, 8, "contiguous", 700),
    (1, 2, 4 * 256, 128, 4, "contiguous", 4 * 256),  # a window of N: plain causal
    # tile ranges that start well inside the block (first loop index 1 to 3):
    # the producer's stage-release waits count each tile's own uses
    (1, 2, 4 * 512, 128, 4, "contiguous", 300),
    (1, 2, 4 * 1024, 128, 4, "striped", 1500),
    (1, 2, 2 * 1024, 64, 2, "contiguous", 333),
]


@pytest.mark.parametrize("case", WINDOW_CASES, ids=lambda c: "B{}H{}N{}d{}P{}{}W{}".format(*c[:5], c[5][0], c[6]))
def test_fwd_sliding_window(case):
    """Causal sliding window (RING_OPT_WINDOW): every row against the
    oracle's windowed dense attention, and the three rotation modes bit for
    bit (with a window the sent tiles can sit inside or below a tile pair's
    key range; they are loaded again at the end)."""
    B, H, N, d, P, layout, W = case
    q, k, v = make_qkv(B, H, N, d, seed=N + W)
    out, lse = run_fwd(B, H, N, d, P, True, layout, q, k, v, rotation=2, window=W)
    BH = B * H
    ref_out, ref_lse = oracle.default().dense(flat(q, BH), flat(k, BH), flat(v, BH), True, window=W)
    d_out, d_lse = report(f"window {case}", out.double().numpy().reshape(BH, N, d),
                          lse.double().numpy().reshape(BH, N), ref_out, ref_lse)
    assert d_out <= TOL_OUT and d_lse <= TOL_LSE
    for mode in (0, 1):
        got = run_fwd(B, H, N, d, P, True, layout, q, k, v, rotation=mode, window=W)
        assert torch.equal(got[0], out) and torch.equal(got[1], lse), mode


@pytest.mark.parametrize("layout", ["contiguous", "striped"])
def test_block_partial_window(layout):
    """Block partials with a window against the oracle's windowed block
    partials, every block of a small ring."""
    B, H, n, d, P, W = 1, 2, 328, 128, 3, 200
    N = n * P
    q, k, v = make_qkv(B, H, N, d, seed=123)
    att = ra.RingAttention(B, H, N, d, P, causal=True, layout=layout)
    att.set_option(ra.RING_OPT_WINDOW, W)
    orc = oracle.default()
    L = lid(layout)
    BH = B * H
    qf, kf, vf = flat(q, BH), flat(k, BH), flat(v, BH)
    worst_o = worst_l = 0.0
    for r in range(P):
        pos_r = [orc.position(L, n, P, r, i) for i in range(n)]
        q_sh = qf[:, pos_r].contiguous()
        for s in range(P):
            j = orc.block_at(P, r, s)
            pos_j = [orc.position(L, n, P, j, i) for i in range(n)]
            k_bl, v_bl = kf[:, pos_j].contiguous(), vf[:, pos_j].contiguous()
            st = att.new_state()
            for x in st:
                x.fill_(float("nan"))
            att.block_partial(r, s, q_sh.reshape(B, H, n, d).cuda(), k_bl.reshape(B, H, n, d).cuda(),
                              v_bl.reshape(B, H, n, d).cuda(), st, 0)
            att.check()
            m, l, o = (x.cpu().double().numpy().reshape(BH * n, -1) for x in st)
            m, l = m[:, 0], l[:, 0]
            rm, rl, ro = orc.block_partial(q_sh, k_bl, v_bl, P, True, L, r, j, window=W)
            rm, rl, ro = rm.reshape(-1), rl.reshape(-1), ro.reshape(BH * n, d)
            empty = np.isneginf(rm)
            assert np.all(np.isneginf(m[empty])) and np.all(l[empty] == 0) and np.all(o[empty] == 0), (r, s)
            ne = ~empty
            if ne.any():
                dl = np.abs((m[ne] + np.log(l[ne])) - (rm[ne] + np.log(rl[ne])))
                do = np.abs(o[ne] / l[ne][:, None] - ro[ne] / rl[ne][:, None])
                worst_l, worst_o = max(worst_l, float(dl.max())), max(worst_o, float(do.max()))
    print(f"block partial window {layout}: max|dout|={worst_o:.3e} max|dlse|={worst_l:.3e}")
    assert worst_o <= TOL_OUT and worst_l <= TOL_LSE
    att.close()


def test_fwd_128k_gqa_sampled():
    _sampled_check(WORKLOADS["gqa-128k"], 256, ring_rows=16)


GQA_CASES = [
    # (B, H, Hkv, N, d, P, causal, layout)
    (1, 4, 2, 4 * 256, 64, 4, True, "striped"),
    (2, 6, 1, 3 * 200, 128, 3, True, "contiguous"),  # multi-query, ragged shards
    (1, 8, 2, 8 * 256, 128, 8, True, "zigzag"),
    (1, 4, 1, 2 * 256, 128, 2, False, "striped"),
]


@pytest.mark.parametrize("case", GQA_CASES, ids=lambda c: "B{}H{}kv{}N{}d{}P{}{}{}".format(
    c[0], c[1], c[2], c[3], c[4], c[5], "c" if c[6] else "n", c[7][0]))
def test_fwd_grouped_query(case):
    """Grouped-query / multi-query attention: H query heads over Hkv K/V
    heads (query head h reads K/V head h / (H/Hkv)).  Against the oracle on
    the K/V heads repeated per query head, and the three rotation modes bit
    for bit (one query head of each group sends the shared block)."""
    B, H, Hkv, N, d, P, causal, layout = case
    q, k, v = make_qkv(B, H, N, d, seed=N + H + Hkv, Hkv=Hkv)
    assert k.shape[1] == Hkv
    out, lse = run_fwd(B, H, N, d, P, causal, layout, q, k, v, rotation=2)
    BH = B * H
    ref_out, ref_lse = oracle.default().dense(flat(q, BH), flat(expand_kv(k, H), BH), flat(expand_kv(v, H), BH),
                                              causal)
    d_out, d_lse = report(f"gqa {case}", out.double().numpy().reshape(BH, N, d), lse.double().numpy().reshape(BH, N),
                          ref_out, ref_lse)
    assert d_out <= TOL_OUT and d_lse <= TOL_LSE
    for mode in (0, 1):
        got = run_fwd(B, H, N, d, P, causal, layout, q, k, v, rotation=mode)
        assert torch.equal(got[0], out) and torch.equal(got[1], lse), mode


def test_block_partial_grouped_query():
    """ring_attn_block_partial with K/V blocks of Hkv heads, accumulated over
    the ring and finalized, equals dense attention on the repeated heads."""
    B, H, Hkv, n, d, P = 2, 4, 2, 256, 128, 3
    N = n * P
    q, k, v = make_qkv(B, H, N, d, seed=91, Hkv=Hkv)
    att = ra.RingAttention(B, H, N, d, P, causal=True, layout="striped", kv_heads=Hkv)
    orc = oracle.default()
    L = LAYOUT_STRIPED
    out = torch.empty((B, H, N, d), device="cuda")
    lse = torch.empty((B, H, N), device="cuda")
    for r in range(P):
        pos_r = [orc.position(L, n, P, r, i) for i in range(n)]
        st = att.new_state()
        att.state_init(st)
        for s in range(P):
            j = orc.block_at(P, r, s)
            pos_j = [orc.position(L, n, P, j, i) for i in range(n)]
            att.block_partial(r, s, q[:, :, pos_r].contiguous().cuda(), k[:, :, pos_j].contiguous().cuda(),
                              v[:, :, pos_j].contiguous().cuda(), st, 1)
        att.finalize(r, st, out, lse)
    att.check()
    BH = B * H
    ref_out, ref_lse = orc.dense(flat(q, BH), flat(expand_kv(k, H), BH), flat(expand_kv(v, H), BH), True)
    d_out, d_lse = report("block ring gqa", out.cpu().double().numpy().reshape(BH, N, d),
                          lse.cpu().double().numpy().reshape(BH, N), ref_out, ref_lse)
    assert d_out <= TOL_OUT and d_lse <= TOL_LSE
    att.close()


@pytest.mark.slow
def test_fwd_1m_striped_sampled():
    _sampled_check(WORKLOADS["striped-1m"], 256)


def test_timing_report():
    B, H, N, d, P = 1, 4, 8 * 512, 128, 8
    q, k, v = make_qkv(B, H, N, d, seed=9)
    att = ra.RingAttention(B, H, N, d, P, causal=True, layout="striped")
    att.set_option(ra.RING_OPT_TIMING, 1)
    for mode in (1, 2):
        att.set_option(ra.RING_OPT_ROTATION, mode)
        att.fwd(q.cuda(), k.cuda(), v.cuda())
        t = att.timing()
        att.check()
        assert len(t["kernel_ms"]) == P and all(x > 0 for x in t["kernel_ms"])
        if mode == 1:
            assert t["copy_ms"][0] == 0 and all(x > 0 for x in t["copy_ms"][1:])
        else:  # striped: every shard has work every step, the kernels send everything
            assert all(x == 0 for x in t["copy_ms"]) and all(x == 0 for x in t["wait_ms"])
        assert all(x >= 0 for x in t["wait_ms"]) and t["pack_ms"] > 0
    att.close()


def test_bad_alignment_is_rejected():
    B, H, N, d, P = 1, 1, 256, 64, 2
    att = ra.RingAttention(B, H, N, d, P, causal=True, layout="striped")
    buf = torch.zeros(B * H * N * d + 8, dtype=torch.bfloat16, device="cuda")
    q = buf[1:1 + B * H * N * d].view(B, H, N, d)  # 2-byte offset: not 16-byte aligned
    out = torch.empty((B, H, N, d), device="cuda")
    lse = torch.empty((B, H, N), device="cuda")
    with pytest.raises(ra.RingAttnError) as e:
        ra.ring_attn_fwd(att.handle, q, q, q, out, lse, att.workspace())
    assert e.value.status == ra._lib.RING_ERR_INVALID_ARG
    att.close()


def test_timing_means_over_calls():
    """The timings are means over the forwards timed since the previous read:
    reading does not clear them, and the first timed call after a read starts
    a new record."""
    B, H, N, d, P = 1, 2, 8 * 512, 128, 8
    q, k, v = (x.cuda() for x in make_qkv(B, H, N, d, seed=9))
    att = ra.RingAttention(B, H, N, d, P, causal=True, layout="striped")
    att.set_option(ra.RING_OPT_TIMING, 1)
    for _ in range(3):
        att.fwd(q, k, v)
    t1 = att.timing()
    t2 = att.timing()
    att.check()
    assert t1 == t2 and all(x > 0 for x in t1["kernel_ms"])
    # one call with side-stream copies (mode 1), then one with the kernels
    # sending (striped: every shard has work every step, so no copies): the
    # first call's copies are in the means
    att.set_option(ra.RING_OPT_ROTATION, 1)
    att.fwd(q, k, v)
    att.set_option(ra.RING_OPT_ROTATION, 2)
    att.fwd(q, k, v)
    t3 = att.timing()
    assert t3["copy_ms"][0] == 0 and all(x > 0 for x in t3["copy_ms"][1:])
    # after the read, a new record holds the last call alone
    att.fwd(q, k, v)
    t4 = att.timing()
    att.check()
    assert all(x == 0 for x in t4["copy_ms"]) and all(x == 0 for x in t4["wait_ms"])
    assert all(x > 0 for x in t4["kernel_ms"]) and t4["pack_ms"] > 0
    att.close()


def test_fwd_heads_beyond_one_grid_dimension():
    """B*H = 65537, an odd count: the step kernel's grid holds at most 65535
    head groups in y (one head each when B*H is odd), so the launch is split
    by heads; heads on both sides of the split match the oracle."""
    B, H, N, d, P = 1, 65537, 128, 64, 1
    q, k, v = make_qkv(B, H, N, d, seed=21)
    att = ra.RingAttention(B, H, N, d, P, causal=True, layout="contiguous")
    out, lse = att.fwd(q.cuda(), k.cuda(), v.cuda())
    att.check()
    torch.cuda.synchronize()
    heads = [0, 65533, 65534, 65535, 65536]
    got_out = out[0, heads].cpu().double().numpy()
    got_lse = lse[0, heads].cpu().double().numpy()
    att.close()
    ref_out, ref_lse = oracle.default().dense(q[0, heads], k[0, heads], v[0, heads], True)
    d_out, d_lse = report("65537 heads", got_out, got_lse, ref_out, ref_lse)
    assert d_out <= TOL_OUT and d_lse <= TOL_LSE
