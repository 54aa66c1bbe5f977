"""Split-K/V decode and short-query prefill (ring_attn_decode) against the
oracle, element by element (GPU only).

Lq new queries sit at global positions N-Lq .. N-1 and see the cached keys
up to their own position under the causal mask.  The oracle is the plain
definition: dense attention of those rows (a full-length query tensor that
holds them at those positions), with grouped K/V heads repeated per query
head.  Tolerances as the ring forward: max|d out| <= 1e-2, max|d lse| <= 1e-3."""
import numpy as np
import pytest
import torch

import oracle
import ring_sequence_parallelism_gb300 as ra
from ring_sequence_parallelism_gb300.inputs import WORKLOADS, expand_kv, make_qkv, make_workload

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


def decode_reference(q, k, v, causal, window=0):
    """Dense rows N-Lq .. N-1 of the oracle for queries q [B, H, Lq, d]."""
    B, H, Lq, d = q.shape
    N = k.shape[2]
    q_full = torch.zeros((B, H, N, d), dtype=torch.bfloat16)
    q_full[:, :, N - Lq:] = q
    BH = B * H
    k, v = expand_kv(k, H), expand_kv(v, H)
    rows = np.arange(N - Lq, N)
    return oracle.default().dense(q_full.reshape(BH, N, d), k.reshape(BH, N, d), v.reshape(BH, N, d), causal,
                                  rows=rows, window=window)


def check(B, H, Hkv, N, d, P, causal, layout, Lq, seed, window=0):
    q_all, k, v = make_qkv(B, H, N, d, seed=seed, Hkv=Hkv)
    q = q_all[:, :, :Lq].contiguous()  # any Lq rows serve as the new queries
    att = ra.RingAttention(B, H, N, d, P, causal=causal, layout=layout, kv_heads=Hkv)
    if window:
        att.set_option(ra.RING_OPT_WINDOW, window)
    out, lse = att.decode(q.cuda(), k.cuda(), v.cuda())
    att.check()
    torch.cuda.synchronize()
    ref_out, ref_lse = decode_reference(q, k, v, causal, window)
    BH = B * H
    d_out = float(np.max(np.abs(out.cpu().double().numpy().reshape(BH, Lq, d) - ref_out)))
    d_lse = float(np.max(np.abs(lse.cpu().double().numpy().reshape(BH, Lq) - ref_lse)))
    print(f"decode B{B} H{H}/{Hkv} N{N} d{d} P{P} {'c' if causal else 'n'} {layout} Lq={Lq}: "
          f"max|dout|={d_out:.3e} max|dlse|={d_lse:.3e}")
    assert d_out <= TOL_OUT and d_lse <= TOL_LSE
    att.close()


CASES = [
    # (B, H, Hkv, N, d, P, causal, layout, Lq)
    (1, 2, 2, 4 * 256, 64, 4, True, "contiguous", 1),
    (1, 2, 2, 4 * 256, 128, 4, True, "striped", 1),
    (2, 3, 3, 3 * 200, 128, 3, True, "striped", 7),       # ragged shards
    (1, 2, 2, 4 * 256, 128, 4, True, "contiguous", 128),
    (1, 2, 2, 4 * 256, 128, 4, True, "striped", 129),     # two query tiles, the second nearly empty
    (1, 2, 2, 3 * 328, 64, 3, True, "contiguous", 300),
    (1, 4, 2, 8 * 256, 128, 8, True, "striped", 64),       # grouped-query
    (1, 4, 1, 2 * 256, 128, 2, False, "striped", 33),      # multi-query, no mask
    (1, 2, 2, 4 * 128, 128, 4, True, "striped", 4 * 128),  # Lq = N: the whole causal attention
    (1, 1, 1, 512, 64, 1, True, "contiguous", 5),          # one shard
    # a few queries: the keys cut into several pieces (the key split)
    (1, 4, 2, 8 * 256, 128, 8, True, "striped", 2),        # grouped-query
    (2, 3, 3, 3 * 200, 64, 3, True, "contiguous", 3),      # ragged shards, B = 2
    (1, 4, 1, 2 * 256, 128, 2, False, "striped", 4),       # multi-query, no mask
    (1, 2, 2, 4 * 256, 128, 4, True, "zigzag", 2),
    (1, 1, 1, 256, 128, 1, True, "contiguous", 1),         # one shard, one query
    (1, 2, 2, 2000, 128, 4, True, "striped", 1),           # 4 pieces, the last key tile ragged (80 keys)
    (1, 2, 2, 2000, 64, 4, True, "contiguous", 130),       # two query tiles, ragged last key tile
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}kv{}N{}d{}P{}{}{}L{}".format(
    c[0], c[1], c[2], c[3], c[4], c[5], "c" if c[6] else "n", c[7][0], c[8]))
def test_decode_matches_oracle(case):
    B, H, Hkv, N, d, P, causal, layout, Lq = case
    check(B, H, Hkv, N, d, P, causal, layout, Lq, seed=N + Lq + H)


@pytest.mark.parametrize("layout,window,Lq", [("contiguous", 100, 1), ("striped", 300, 64), ("striped", 129, 200),
                                              ("contiguous", 1000, 300), ("striped", 300, 3)])
def test_decode_sliding_window(layout, window, Lq):
    """Decode with a causal sliding window: each new query sees the last
    `window` positions up to its own."""
    check(1, 2, 2, 4 * 256, 128, 4, True, layout, Lq, seed=Lq + window, window=window)


@pytest.mark.parametrize("Lq", [1, 128])
def test_decode_128k_workload(Lq):
    """The 128K striped workload's cache (16 heads, 1% of key rows x8), one
    decode token and a 128-token prefill chunk, every row."""
    w = WORKLOADS["striped-128k"]
    q_all, k, v = make_workload(w)
    q = q_all[:, :, :Lq].contiguous()
    att = ra.RingAttention(w.B, w.H, w.N, w.d, w.P, causal=True, layout=w.layout)
    out, lse = att.decode(q.cuda(), k.cuda(), v.cuda())
    att.check()
    torch.cuda.synchronize()
    ref_out, ref_lse = decode_reference(q, k, v, True)
    BH = w.B * w.H
    d_out = float(np.max(np.abs(out.cpu().double().numpy().reshape(BH, Lq, w.d) - ref_out)))
    d_lse = float(np.max(np.abs(lse.cpu().double().numpy().reshape(BH, Lq) - ref_lse)))
    print(f"decode striped-128k Lq={Lq}: max|dout|={d_out:.3e} max|dlse|={d_lse:.3e}")
    assert d_out <= TOL_OUT and d_lse <= TOL_LSE
    att.close()


def test_decode_layout_independent():
    """The cache is read in natural order and cut into the same key pieces
    whatever the handle's layout and P: every layout gives the same bits."""
    B, H, N, d, Lq = 1, 4, 4096, 128, 3
    q_all, k, v = make_qkv(B, H, N, d, seed=733)
    q, k, v = q_all[:, :, :Lq].contiguous().cuda(), k.cuda(), v.cuda()
    got = []
    for layout, P in (("contiguous", 4), ("striped", 4), ("zigzag", 4), ("striped", 8), ("contiguous", 1)):
        att = ra.RingAttention(B, H, N, d, P, causal=True, layout=layout)
        out, lse = att.decode(q, k, v)
        att.check()
        got.append((out.cpu(), lse.cpu()))
        att.close()
    for out, lse in got[1:]:
        assert torch.equal(out, got[0][0]) and torch.equal(lse, got[0][1])


def test_decode_rejects_bad_lengths():
    """Lq must lie in [1, N] (zigzag decode is covered in
    tests/test_gpu_zigzag_masks.py)."""
    k, v = (torch.zeros((1, 1, 512, 64), dtype=torch.bfloat16, device="cuda") for _ in range(2))
    att = ra.RingAttention(1, 1, 512, 64, 2, causal=True, layout="striped")
    q = torch.zeros((1, 1, 513, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ra.RingAttnError):
        att.decode(q, k, v)
    att.close()
