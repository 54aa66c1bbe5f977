"""The 128K striped workload (B=1, H=16, N=131072, d=128, P=16, causal, 1%
of key rows x8) against the float64 oracle on two whole heads (GPU only,
slow: the oracle's dense forward of one head is about 4.4e12 float64 FLOPs,
close to two minutes on 16 host cores).

Forward: every one of the 131072 rows of heads 0 and 15, out and lse,
within max|d out| <= 1e-2 and max|d lse| <= 1e-3 (the other 14 heads are
checked on 256 sampled rows plus the shard and chunk edges in
test_gpu_parity.py).  Backward: dK and dV at keys that almost every query
sees (0, 1, a shard's last, the next shard's first, the middle of the
sequence, eight seeded ones) and at the last key, for the same two heads,
against the oracle's gradients from its own forward statistics, under the
bounds of test_gpu_backward.py (relative L2 <= 1e-2, largest element error
<= 1e-2 of the largest magnitude).  Every call goes through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import ring_sequence_parallelism_gb300 as ra
from ring_sequence_parallelism_gb300.inputs import WORKLOADS, make_dout, make_workload

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

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


def test_128k_striped_two_whole_heads():
    w = WORKLOADS["striped-128k"]
    q, k, v = make_workload(w)
    do = make_dout(w.B, w.H, w.N, w.d, w.seed)
    att = ra.RingAttention(w.B, w.H, w.N, w.d, w.P, causal=w.causal, layout=w.layout)
    qc, kc, vc, doc = (x.cuda() for x in (q, k, v, do))
    out, lse = att.fwd(qc, kc, vc)
    dq, dk, dv = att.bwd(qc, kc, vc, out, lse, doc)
    att.check()
    torch.cuda.synchronize()
    BH = w.B * w.H
    heads = [0, w.H - 1]
    flat = lambda t: t.reshape(BH, w.N, w.d)
    sel = lambda t: flat(t)[heads].contiguous()
    got_out = sel(out.cpu()).double().numpy()
    got_lse = lse.cpu().reshape(BH, w.N)[heads].double().numpy()
    got_dk, got_dv = sel(dk.cpu()).double().numpy(), sel(dv.cpu()).double().numpy()
    del qc, kc, vc, doc, out, lse, dq, dk, dv
    att.close()

    orc = oracle.default()
    ref_out, ref_lse = orc.dense(sel(q), sel(k), sel(v), True)
    d_out = float(np.max(np.abs(got_out - ref_out)))
    d_lse = float(np.max(np.abs(got_lse - ref_lse)))
    print(f"striped-128k heads {heads}, all {w.N} rows: max|dout|={d_out:.3e} max|dlse|={d_lse:.3e}")
    assert d_out <= TOL_OUT and d_lse <= TOL_LSE

    n = w.n
    g = np.random.default_rng(2005)
    keys = sorted(set([0, 1, n - 1, n, w.N // 2, w.N - 1] + g.choice(w.N, 8, replace=False).tolist()))
    rk, rv = orc.dense_bwd_keys(sel(q), sel(k), sel(v), sel(do), ref_out, ref_lse, True, keys)
    for name, a, b in (("dk", got_dk[:, keys], rk), ("dv", got_dv[:, keys], rv)):
        err = np.abs(a - b)
        rel2 = float(np.linalg.norm(a - b) / np.linalg.norm(b))
        rmax = float(err.max() / np.abs(b).max())
        print(f"striped-128k backward {name} at keys {keys}: rel L2 {rel2:.2e}, max {err.max():.2e} "
              f"({rmax:.2e} of max|ref|)")
        assert rel2 <= TOL_REL_L2 and rmax <= TOL_MAX, (name, rel2, rmax)
