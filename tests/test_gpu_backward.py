"""The ring backward (CUDA, through the C ABI) against the float64 oracle.

The gradients have no stated tolerance; this one follows from the
arithmetic.  The kernels take the forward's fp32 out and lse, recompute S
in fp32 on the tensor cores, and round P (the dV operand) and dS (the dK and
dQ operand) to bf16 (unit roundoff u = 2^-9), accumulating in fp32.  A
float64 model of exactly that rounding on N(0, 1) inputs (N = 512..4096,
d = 64 and 128, causal and not) gives a relative L2 error of 1.5-2.2e-3 and
a largest element error of 1.2e-3 to 8.1e-3 times the tensor's largest
magnitude; the GPU measures 0.9e-3 to 3.2e-3 on the cases below.  The
bounds, for each of dq, dk and dv (the second 1.2 times the model's worst):
    ||got - ref||_2 <= 1e-2 ||ref||_2   and   max|got - ref| <= 1e-2 max|ref|.
Where the reference is exactly zero (a window of one token: P = 1, so dQ
and dK vanish), what remains is dS = P (dP - D) with dP = dO . v from the
tensor cores and D = dO . out from the preprocessing, two fp32 evaluations
of the same d-term dot product: |dP - D| is a few ulps of sum |dO_c v_c|
(about 1e-5 at d = 128), so the bound there is max|got| <= 1e-3.
Every call goes through the C ABI (the ctypes binding); the oracle computes
its gradients from the inputs alone (none of its inputs come from the GPU).
"""
import numpy as np
import pytest
import torch

import oracle
import ring_sequence_parallelism_gb300 as ra
from ring_sequence_parallelism_gb300.inputs import WORKLOADS, make_dout, make_qkv, make_workload, sample_rows

pytestmark = pytest.mark.gpu

TOL_REL_L2 = 1e-2
TOL_MAX = 1e-2
TOL_ZERO_REF = 1e-3


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from ring_sequence_parallelism_gb300 import build

    build.build()
    ra._lib.load()


def check_grads(name, got, ref):
    worst = []
    for g_name, a, b in zip(("dq", "dk", "dv"), got, ref):
        a = np.asarray(a, np.float64)
        b = np.asarray(b, np.float64)
        err = np.abs(a - b)
        if not np.any(b):
            worst.append(f"{g_name}: reference 0, max|got| {err.max():.2e}")
            assert err.max() <= TOL_ZERO_REF, f"{name} {g_name}: max|got| {err.max():.3e} > {TOL_ZERO_REF} (reference 0)"
            continue
        rel2 = float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))
        rmax = float(err.max() / max(np.abs(b).max(), 1e-300)) if err.size else 0.0
        worst.append(f"{g_name}: rel L2 {rel2:.2e}, max {err.max():.2e} ({rmax:.2e} of max|ref|)")
        assert rel2 <= TOL_REL_L2, f"{name} {g_name}: relative L2 error {rel2:.3e} > {TOL_REL_L2}"
        assert rmax <= TOL_MAX, f"{name} {g_name}: max error {rmax:.3e} of max|ref| > {TOL_MAX}"
    print(f"{name}: " + "; ".join(worst))


def gpu_fwd_bwd(B, H, N, d, P, causal, layout, q, k, v, do, window=0, lap=None, kv_heads=None, segments=None):
    """Forward then backward through the C ABI; lap None keeps the library's
    default schedule (RING_OPT_BWD_LAP), True/False sets it."""
    att = ra.RingAttention(B, H, N, d, P, causal=causal, layout=layout, kv_heads=kv_heads)
    if window:
        att.set_option(ra.RING_OPT_WINDOW, window)
    if segments is not None:
        att.set_segments(segments)
    if lap is not None:
        att.set_option(ra.RING_OPT_BWD_LAP, 1 if lap else 0)
    qc, kc, vc, doc = (x.cuda() for x in (q, k, v, do))
    out, lse = att.fwd(qc, kc, vc)
    dq, dk, dv = att.bwd(qc, kc, vc, out, lse, doc)
    att.check()
    torch.cuda.synchronize()
    res = tuple(x.cpu() for x in (dq, dk, dv))
    att.close()
    return res


CASES = [
    # (B, H, N, d, P, causal, layout, window)
    (1, 2, 512, 64, 4, False, "contiguous", 0),  # the 512-token non-causal workload's shape
    (1, 2, 512, 64, 4, True, "contiguous", 0),
    (1, 2, 512, 64, 4, True, "striped", 0),
    (1, 2, 1024, 128, 8, True, "striped", 0),
    (1, 2, 1024, 128, 8, False, "striped", 0),
    (1, 2, 1024, 128, 1, True, "contiguous", 0),  # P = 1: one step, no ring
    (1, 2, 2624, 128, 8, True, "contiguous", 0),  # n = 328: ragged last tile
    (1, 2, 2624, 128, 8, True, "striped", 0),
    (1, 1, 1000, 128, 8, True, "striped", 0),  # n = 125: a single partial tile
    (2, 1, 768, 64, 3, True, "contiguous", 0),  # B = 2, odd P
    (1, 2, 2048, 128, 4, True, "striped", 300),  # sliding window
    (1, 2, 2048, 128, 4, True, "contiguous", 300),
    (1, 2, 1024, 128, 4, True, "striped", 1),  # window 1: each query sees itself only
]


@pytest.mark.parametrize("B,H,N,d,P,causal,layout,window", CASES,
                         ids=[f"{c[6]}-N{c[2]}-d{c[3]}-P{c[4]}-{'c' if c[5] else 'nc'}-w{c[7]}" for c in CASES])
def test_bwd_small(orc, B, H, N, d, P, causal, layout, window):
    q, k, v = make_qkv(B, H, N, d, seed=500 + N + P)
    do = make_dout(B, H, N, d, seed=500 + N + P)
    got = gpu_fwd_bwd(B, H, N, d, P, causal, layout, q, k, v, do, window)
    BH = B * H
    ref = orc.dense_bwd(q.reshape(BH, N, d), k.reshape(BH, N, d), v.reshape(BH, N, d), do.reshape(BH, N, d),
                        causal, window=window)
    check_grads(f"bwd {layout} N={N} d={d} P={P} causal={causal} w={window}",
                [g.reshape(BH, N, d).numpy() for g in got], ref)


@pytest.mark.parametrize("name", ["contiguous-8k", "striped-8k"])
def test_bwd_8k(orc, name):
    """The two 8K workloads in full, element by element."""
    w = WORKLOADS[name]
    q, k, v = make_workload(w)
    do = make_dout(w.B, w.H, w.N, w.d, w.seed)
    got = gpu_fwd_bwd(w.B, w.H, w.N, w.d, w.P, w.causal, w.layout, q, k, v, do)
    BH = w.B * w.H
    flat = lambda t: t.reshape(BH, w.N, w.d)
    ref = orc.dense_bwd(flat(q), flat(k), flat(v), flat(do), w.causal)
    check_grads(f"bwd {name}", [flat(g).numpy() for g in got], ref)


def test_bwd_layouts_agree():
    """Contiguous and striped shards give the same gradients (the layout
    only changes which tokens each shard holds), up to rounding order."""
    B, H, N, d, P = 1, 2, 2048, 128, 8
    q, k, v = make_qkv(B, H, N, d, seed=77)
    do = make_dout(B, H, N, d, seed=77)
    a = gpu_fwd_bwd(B, H, N, d, P, True, "contiguous", q, k, v, do)
    b = gpu_fwd_bwd(B, H, N, d, P, True, "striped", q, k, v, do)
    check_grads("contiguous vs striped", [x.numpy() for x in b], [x.numpy() for x in a])


def test_bwd_128k_sampled(orc):
    """The 128K striped workload (1% of key rows x8): dQ at 256 sampled
    query rows per head for 2 heads, dK and dV at four late keys (cheap for
    the oracle under the causal mask), and for every head the gradient
    identities sum_k dK_k = 0 and sum_k dV_k = sum_t dO_t, each within 1e-2
    of the sum of magnitudes (the relative bound above)."""
    w = WORKLOADS["striped-128k"]
    q, k, v = make_workload(w)
    do = make_dout(w.B, w.H, w.N, w.d, w.seed)
    dq, dk, dv = gpu_fwd_bwd(w.B, w.H, w.N, w.d, w.P, w.causal, w.layout, q, k, v, do)
    BH = w.B * w.H
    flat = lambda t: t.reshape(BH, w.N, w.d)
    dq, dk, dv, dof = flat(dq).double(), flat(dk).double(), flat(dv).double(), flat(do).double()
    # identities, every head
    s_dk = dk.sum(1)
    assert bool((s_dk.abs() <= 1e-2 * dk.abs().sum(1)).all()), "sum_k dK_k = 0 violated"
    s_dv = dv.sum(1) - dof.sum(1)
    assert bool((s_dv.abs() <= 1e-2 * dv.abs().sum(1)).all()), "sum_k dV_k = sum_t dO_t violated"
    # sampled rows, two heads
    heads = [0, w.H - 1]
    qrows = sample_rows(w.N, 256, extra=(0, 1, w.N // 2, w.N - 1)).numpy()
    krows = np.array([w.N - 1, w.N - 2, w.N - 5, w.N - 17])
    sel = lambda t: flat(t)[heads].contiguous()
    rq, rk, rv = orc.dense_bwd_rows(sel(q), sel(k), sel(v), sel(do), True, qrows, krows)
    got = (dq[heads][:, qrows].numpy(), dk[heads][:, krows].numpy(), dv[heads][:, krows].numpy())
    check_grads("bwd striped-128k sampled", got, (rq, rk, rv))


@pytest.mark.parametrize("layout,window", [("striped", 0), ("contiguous", 0), ("striped", 300)])
def test_bwd_grouped_query(orc, layout, window):
    """Grouped-query attention (8 query heads over 2 K/V heads): dQ per
    query head, and dK, dV per K/V head, which reads as G = 4 query heads'
    copies of one tensor, so its gradient is the sum of the copies'
    gradients (the oracle runs on K/V repeated per query head)."""
    from ring_sequence_parallelism_gb300.inputs import expand_kv

    B, H, Hkv, N, d, P = 1, 8, 2, 2048, 128, 4
    G = H // Hkv
    q, k, v = make_qkv(B, H, N, d, seed=660, Hkv=Hkv)
    do = make_dout(B, H, N, d, seed=660)
    att = ra.RingAttention(B, H, N, d, P, causal=True, layout=layout, kv_heads=Hkv)
    if window:
        att.set_option(ra.RING_OPT_WINDOW, window)
    qc, kc, vc, doc = (x.cuda() for x in (q, k, v, do))
    out, lse = att.fwd(qc, kc, vc)
    dq, dk, dv = att.bwd(qc, kc, vc, out, lse, doc)
    att.check()
    att.close()
    flat = lambda t: t.reshape(-1, N, d)
    rq, rk, rv = orc.dense_bwd(flat(q), flat(expand_kv(k, H)), flat(expand_kv(v, H)), flat(do), True, window=window)
    rk = rk.reshape(B * Hkv, G, N, d).sum(1)
    rv = rv.reshape(B * Hkv, G, N, d).sum(1)
    check_grads(f"bwd gqa {layout} w={window}", [flat(g).cpu().numpy() for g in (dq, dk, dv)], (rq, rk, rv))


@pytest.mark.parametrize("P,causal", [(4, True), (2, True), (4, False), (1, True)])
def test_bwd_zigzag(orc, P, causal):
    """The zigzag layout (2P chunks, shard r holding chunks r and 2P-1-r):
    every gradient element against the oracle."""
    B, H, d = 1, 2, 128
    N = 2 * P * 256  # chunks of 256 tokens
    q, k, v = make_qkv(B, H, N, d, seed=670 + P)
    do = make_dout(B, H, N, d, seed=670 + P)
    got = gpu_fwd_bwd(B, H, N, d, P, causal, "zigzag", q, k, v, do)
    flat = lambda t: t.reshape(B * H, N, d)
    ref = orc.dense_bwd(flat(q), flat(k), flat(v), flat(do), causal)
    check_grads(f"bwd zigzag P={P} causal={causal}", [flat(g).numpy() for g in got], ref)


def test_bwd_zigzag_8k(orc):
    """The 8K workload in the zigzag layout, in full."""
    w = WORKLOADS["zigzag-8k"]
    q, k, v = make_workload(w)
    do = make_dout(w.B, w.H, w.N, w.d, w.seed)
    got = gpu_fwd_bwd(w.B, w.H, w.N, w.d, w.P, w.causal, w.layout, q, k, v, do)
    flat = lambda t: t.reshape(w.B * w.H, w.N, w.d)
    ref = orc.dense_bwd(flat(q), flat(k), flat(v), flat(do), w.causal)
    check_grads("bwd zigzag-8k", [flat(g).numpy() for g in got], ref)


LAP_CASES = [
    # (B, H, Hkv, N, d, P, causal, layout, window, segments)
    (1, 2, 2, 1024, 128, 8, True, "striped", 0, None),
    (1, 2, 2, 1024, 64, 4, False, "contiguous", 0, None),
    (1, 2, 2, 2624, 128, 8, True, "contiguous", 0, None),  # n = 328: ragged last tile
    (1, 2, 2, 2048, 128, 4, True, "zigzag", 0, None),
    (1, 2, 2, 2048, 128, 4, True, "striped", 300, None),  # sliding window
    (1, 8, 2, 2048, 128, 4, True, "contiguous", 0, None),  # grouped-query: G = 4
    (1, 2, 2, 1024, 128, 4, True, "striped", 0, [0, 100, 101, 613, 1024]),  # packed documents
    (2, 1, 1, 768, 64, 3, True, "contiguous", 0, None),  # B = 2, odd P
]


@pytest.mark.parametrize("case", LAP_CASES,
                         ids=[f"{c[7]}-N{c[3]}-d{c[4]}-P{c[5]}-H{c[1]}/{c[2]}-{'c' if c[6] else 'nc'}-w{c[8]}"
                              f"-s{0 if c[9] is None else len(c[9]) - 1}" for c in LAP_CASES])
def test_bwd_lap(orc, case):
    """RING_OPT_BWD_LAP = 1 (one launch per kernel, every CTA making its
    tile's whole lap with the accumulators in tensor memory) gives exactly
    the gradients of RING_OPT_BWD_LAP = 0 (one launch per ring step; same
    MMAs on the same fp32 values in the same order), and both pass the
    oracle check."""
    from ring_sequence_parallelism_gb300.inputs import expand_kv

    B, H, Hkv, N, d, P, causal, layout, window, segments = case
    q, k, v = make_qkv(B, H, N, d, seed=680 + N + P, Hkv=Hkv)
    do = make_dout(B, H, N, d, seed=680 + N + P)
    args = (B, H, N, d, P, causal, layout, q, k, v, do)
    step = gpu_fwd_bwd(*args, window=window, kv_heads=Hkv, segments=segments, lap=False)
    lap = gpu_fwd_bwd(*args, window=window, kv_heads=Hkv, segments=segments, lap=True)
    for name, a, b in zip(("dq", "dk", "dv"), lap, step):
        assert torch.equal(a, b), f"lap and per-step {name} differ (max {float((a - b).abs().max()):.3e})"
    G = H // Hkv
    flat = lambda t: t.reshape(-1, N, d)
    rq, rk, rv = orc.dense_bwd(flat(q), flat(expand_kv(k, H)), flat(expand_kv(v, H)), flat(do), causal,
                               window=window, segments=segments)
    rk = rk.reshape(B * Hkv, G, N, d).sum(1)
    rv = rv.reshape(B * Hkv, G, N, d).sum(1)
    check_grads(f"bwd lap {case}", [flat(g).numpy() for g in lap], (rq, rk, rv))
    check_grads(f"bwd per-step {case}", [flat(g).numpy() for g in step], (rq, rk, rv))


def test_bwd_lap_128k_sampled(orc):
    """The two schedules on the 128K striped workload give identical
    gradients (every element); the sampled oracle test above checks the
    default one."""
    w = WORKLOADS["striped-128k"]
    q, k, v = make_workload(w)
    do = make_dout(w.B, w.H, w.N, w.d, w.seed)
    args = (w.B, w.H, w.N, w.d, w.P, w.causal, w.layout, q, k, v, do)
    step = gpu_fwd_bwd(*args, lap=False)
    lap = gpu_fwd_bwd(*args, lap=True)
    for name, a, b in zip(("dq", "dk", "dv"), lap, step):
        assert torch.equal(a, b), f"lap and per-step {name} differ (max {float((a - b).abs().max()):.3e})"
