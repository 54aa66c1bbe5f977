"""The ring forward in one launch (RING_OPT_FWD_LAP = 1) against the float64
oracle, through the C ABI (GPU only).

Each CTA owns a pair of query tiles of shard r and meets blocks r, r-1, ..
in step order with the running state on chip; the blocks are read in place.
Every row is compared with the oracle's dense attention under the parity
tolerances (max|d out| <= 1e-2, max|d lse| <= 1e-3), for every layout,
causal or not, ragged shards, grouped K/V heads, sliding windows and packed
documents; the 128K windowed and packed workloads on sampled rows.  The lap
and the step schedule run the same arithmetic per key tile, but not in the
same order of key tiles (the step kernel rotates the order in blocks without
a diagonal, so that the tiles it sends along the ring come last) and the step
schedule stores m between steps in natural-log units; P is rounded to bf16
against a different running maximum, so the two agree within the parity
tolerance, not bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import ring_sequence_parallelism_gb300 as ra
from ring_sequence_parallelism_gb300.inputs import WORKLOADS, expand_kv, make_qkv, make_workload, sample_rows

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


def run(B, H, N, d, P, causal, layout, q, k, v, lap, window=0, bounds=None):
    att = ra.RingAttention(B, H, N, d, P, causal=causal, layout=layout, kv_heads=k.shape[1])
    if window:
        att.set_option(ra.RING_OPT_WINDOW, window)
    if bounds is not None:
        att.set_segments(bounds)
    att.set_option(ra.RING_OPT_FWD_LAP, 1 if lap else 0)
    out, lse = att.fwd(q.cuda(), k.cuda(), v.cuda())
    att.check()
    torch.cuda.synchronize()
    res = out.cpu(), lse.cpu()
    att.close()
    return res


CASES = [
    # (B, H, Hkv, N, d, P, causal, layout, window, bounds)
    (1, 2, 2, 512, 64, 4, False, "contiguous", 0, None),  # the 512-token non-causal workload's shape
    (1, 2, 2, 4 * 512, 128, 4, True, "contiguous", 0, None),  # skipped blocks
    (1, 2, 2, 4 * 512, 128, 4, True, "striped", 0, None),
    (1, 2, 2, 4 * 512, 128, 4, True, "zigzag", 0, None),
    (1, 2, 2, 8 * 768, 128, 8, True, "zigzag", 0, None),  # chunks of 384: tile pair (2, 3) spans two chunks
    (1, 2, 2, 3 * 328, 128, 3, True, "contiguous", 0, None),  # ragged shards, odd P
    (1, 2, 2, 3 * 328, 64, 3, True, "striped", 0, None),
    (1, 1, 1, 8 * 125, 128, 8, True, "striped", 0, None),  # a single partial tile per shard
    (2, 8, 2, 4 * 256, 128, 4, True, "striped", 0, None),  # grouped K/V heads, B = 2
    (1, 4, 1, 2 * 256, 128, 2, False, "striped", 0, None),  # multi-query, non-causal
    (1, 2, 2, 1024, 128, 1, True, "contiguous", 0, None),  # P = 1
    (1, 2, 2, 8 * 256, 128, 8, True, "striped", 700, None),  # sliding windows
    (1, 2, 2, 4 * 512, 128, 4, True, "contiguous", 300, None),
    (1, 2, 2, 4 * 256, 64, 4, True, "contiguous", 1, None),
    (1, 2, 2, 1024, 128, 4, True, "striped", 0, [0, 100, 101, 613, 1024]),  # packed documents
    (1, 2, 2, 4096, 128, 4, True, "contiguous", 0, [0, 1000, 3950, 4096]),
    (1, 2, 2, 1024, 128, 4, False, "contiguous", 0, [0, 128, 1024]),
    (2, 1, 1, 2048, 128, 8, True, "striped", 200, [0, 700, 1500, 2048]),  # window and documents
]


def case_id(c):
    return "B{}H{}kv{}N{}d{}P{}{}{}W{}s{}".format(c[0], c[1], c[2], c[3], c[4], c[5], "c" if c[6] else "n", c[7][0],
                                                  c[8], 0 if c[9] is None else len(c[9]) - 1)


@pytest.mark.parametrize("case", CASES, ids=case_id)
def test_lap_matches_oracle(orc, case):
    B, H, Hkv, N, d, P, causal, layout, window, bounds = case
    q, k, v = make_qkv(B, H, N, d, seed=900 + N + H, Hkv=Hkv)
    BH = B * H
    flat = lambda t: t.reshape(BH, N, -1)
    ref_o, ref_l = orc.dense(flat(q), flat(expand_kv(k, H)), flat(expand_kv(v, H)), causal, window=window,
                             segments=bounds)
    out, lse = run(B, H, N, d, P, causal, layout, q, k, v, True, window, bounds)
    d_out = float(np.max(np.abs(out.double().numpy().reshape(BH, N, d) - ref_o)))
    d_lse = float(np.max(np.abs(lse.double().numpy().reshape(BH, N) - ref_l)))
    step = run(B, H, N, d, P, causal, layout, q, k, v, False, window, bounds)
    s_out = float((out - step[0]).abs().max())
    s_lse = float((lse - step[1]).abs().max())
    print(f"lap {case}: max|dout|={d_out:.3e} max|dlse|={d_lse:.3e}; vs step {s_out:.2e} {s_lse:.2e}")
    assert d_out <= TOL_OUT and d_lse <= TOL_LSE
    assert s_out <= TOL_OUT and s_lse <= TOL_LSE


@pytest.mark.parametrize("name", ["swa-128k", "packed-128k", "striped-128k"])
def test_lap_128k_sampled(orc, name):
    """The 128K workloads (1% of key rows x8) with the lap: 256 seeded rows
    per head plus the shard edges, against the oracle."""
    w = WORKLOADS[name]
    q, k, v = make_workload(w)
    out, lse = run(w.B, w.H, w.N, w.d, w.P, w.causal, w.layout, q, k, v, True, w.window, w.segments())
    BH = w.B * w.H
    rows = sample_rows(w.N, 256, extra=(0, 1, w.n - 1, w.n, w.N // 2, w.N - 1)).numpy()
    ref_o, ref_l = orc.dense(q.reshape(BH, w.N, w.d), k.reshape(BH, w.N, w.d), v.reshape(BH, w.N, w.d), w.causal,
                             rows=rows, window=w.window, segments=w.segments())
    got_o = out.reshape(BH, w.N, w.d)[:, rows].double().numpy()
    got_l = lse.reshape(BH, w.N)[:, rows].double().numpy()
    d_out = float(np.max(np.abs(got_o - ref_o)))
    d_lse = float(np.max(np.abs(got_l - ref_l)))
    print(f"lap {name} ({rows.size} rows/head): max|dout|={d_out:.3e} max|dlse|={d_lse:.3e}")
    assert d_out <= TOL_OUT and d_lse <= TOL_LSE
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()


def test_lap_timing_and_timeout():
    """ring_attn_get_timing reports the single launch in entry 0; a bounded
    wait that nothing completes (the V loads dropped) ends with
    RING_ERR_TIMEOUT and the next call is correct."""
    B, H, N, d, P = 1, 1, 512, 128, 2
    q, k, v = (x.cuda() for x in make_qkv(B, H, N, d, seed=4))
    att = ra.RingAttention(B, H, N, d, P, causal=True, layout="striped")
    att.set_option(ra.RING_OPT_FWD_LAP, 1)
    att.set_option(ra.RING_OPT_TIMING, 1)
    out, lse = att.fwd(q, k, v)
    t = att.timing()
    att.check()
    assert t["kernel_ms"][0] > 0 and all(x < t["kernel_ms"][0] for x in t["kernel_ms"][1:])
    att.set_option(ra.RING_OPT_WAIT_LIMIT_NS, 20_000_000)
    att.set_option(ra.RING_OPT_DEBUG_DROP_V_LOADS, 1)
    att.fwd(q, k, v)
    with pytest.raises(ra.RingAttnError) as e:
        att.check()
    assert e.value.status == ra._lib.RING_ERR_TIMEOUT
    att.set_option(ra.RING_OPT_DEBUG_DROP_V_LOADS, 0)
    att.set_option(ra.RING_OPT_WAIT_LIMIT_NS, 2_000_000_000)
    out2, lse2 = att.fwd(q, k, v)
    att.check()
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    att.close()
