"""Pins that tie the float64 oracle to what the pages and the mathematics fix.

Each pin takes an ``oracle.Oracle`` and raises AssertionError on a mismatch.
They are run against the real oracle (tests/test_oracle.py) and against
copies of it with planted mistakes (tests/test_oracle_mutations.py), which
must each trip at least one pin.

Sources cited by page title and section:
  [GRA]   "GPU Ring Attention" (aicassindra.com)
  [ZQ]    Ring attention explainer page (zenaique.com)
  [RA-CN] "Ring Attention：把超长序列沿设备环流动" (charlestar.github.io)
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

from oracle import LAYOUT_CONTIGUOUS, LAYOUT_STRIPED, LAYOUT_ZIGZAG, bits_to_f64, bf16_bits

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

LAYOUTS = (LAYOUT_CONTIGUOUS, LAYOUT_STRIPED, LAYOUT_ZIGZAG)


def layouts_for(N, P):
    """The layouts a shape admits: zigzag needs N divisible by 2P."""
    return [lay for lay in LAYOUTS if lay != LAYOUT_ZIGZAG or N % (2 * P) == 0]


def rand_bits(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    t = (torch.randn(shape, generator=g, dtype=torch.float32) * scale).to(torch.bfloat16)
    return bf16_bits(t)


def to_bits(x: np.ndarray) -> np.ndarray:
    """float array -> bf16 bits (values must already be bf16-representable)."""
    t = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16)
    back = t.to(torch.float32).numpy()
    assert np.array_equal(back, np.asarray(x, np.float32)), "value not exact in bf16"
    return bf16_bits(t)


def allowed_matrix(N, causal):
    if not causal:
        return np.ones((N, N), bool)
    return np.tril(np.ones((N, N), bool))


def _close(a, b, tol, what):
    err = float(np.max(np.abs(np.asarray(a) - np.asarray(b)))) if np.size(a) else 0.0
    assert err <= tol, f"{what}: max abs err {err:.3e} > {tol:.1e}"


# ---------------------------------------------------------------- dense path
def pin_equal_keys_closed_form(orc):
    """All key rows equal: every allowed key has the same score s, so the
    softmax is uniform: out = mean of the allowed v rows, lse = s + ln(count)."""
    BH, N, d = 2, 24, 8
    q = rand_bits((BH, N, d), 11)
    k0 = rand_bits((BH, 1, d), 12)
    k = np.ascontiguousarray(np.repeat(k0, N, axis=1))
    v = rand_bits((BH, N, d), 13)
    qf, kf, vf = bits_to_f64(q), bits_to_f64(k), bits_to_f64(v)
    for causal in (False, True):
        cnt = np.arange(1, N + 1) if causal else np.full(N, N)
        mean_v = (np.cumsum(vf, axis=1) / cnt[None, :, None]) if causal else np.repeat(vf.mean(1, keepdims=True), N, 1)
        s = np.einsum("bnd,bd->bn", qf, kf[:, 0, :]) / math.sqrt(d)
        exp_lse = s + np.log(cnt)[None, :]
        out, lse = orc.dense(q, k, v, causal)
        _close(out, mean_v, 1e-12, "equal keys: out")
        _close(lse, exp_lse, 1e-12, "equal keys: lse")
        for layout in LAYOUTS:
            out, lse = orc.ring(q, k, v, 4, causal, layout)
            _close(out, mean_v, 1e-12, "equal keys (ring): out")
            _close(lse, exp_lse, 1e-12, "equal keys (ring): lse")


def pin_constant_values(orc):
    """Every v row equal to c: any convex combination is c."""
    BH, N, d = 2, 16, 4
    q, k = rand_bits((BH, N, d), 21), rand_bits((BH, N, d), 22)
    c = np.array([0.5, -1.25, 3.0, 0.0078125], np.float32)
    v = to_bits(np.broadcast_to(c, (BH, N, d)))
    for causal in (False, True):
        out, _ = orc.dense(q, k, v, causal)
        _close(out, np.broadcast_to(c, out.shape), 1e-13, "constant v (dense)")
        out, _ = orc.ring(q, k, v, 4, causal, LAYOUT_STRIPED)
        _close(out, np.broadcast_to(c, out.shape), 1e-13, "constant v (ring)")


def pin_causal_first_row(orc):
    """Causal row 0 sees only key 0: out_0 = v_0 and lse_0 = s_00."""
    BH, N, d = 3, 12, 8
    q, k, v = rand_bits((BH, N, d), 31), rand_bits((BH, N, d), 32), rand_bits((BH, N, d), 33)
    qf, kf, vf = bits_to_f64(q), bits_to_f64(k), bits_to_f64(v)
    s00 = np.einsum("bd,bd->b", qf[:, 0], kf[:, 0]) / math.sqrt(d)
    for fn in (lambda: orc.dense(q, k, v, True),
               lambda: orc.ring(q, k, v, 3, True, LAYOUT_CONTIGUOUS),
               lambda: orc.ring(q, k, v, 3, True, LAYOUT_STRIPED)):
        out, lse = fn()
        _close(out[:, 0], vf[:, 0], 0.0, "causal row 0: out")
        _close(lse[:, 0], s00, 1e-14, "causal row 0: lse")


def pin_dominant_key(orc):
    """One key outscores every other allowed key by ~2000 nats: the output is
    that key's value (scores of 2048, whose exp overflows even float64, also
    test that the oracle subtracts the row max; [RA-CN] "正确性测试应覆盖哪些边界": online
    softmax stability under extreme scores)."""
    BH, N, d = 1, 16, 4
    q = to_bits(np.full((BH, N, d), 32.0, np.float32))
    kv = np.full((BH, N, d), 1.0, np.float32)
    kv[:, 5, :] = 32.0  # q.k/2 = 2048 for key 5, 64 for the others
    k = to_bits(kv)
    v = rand_bits((BH, N, d), 41)
    vf = bits_to_f64(v)
    for causal in (False, True):
        out, lse = orc.dense(q, k, v, causal)
        rows = np.arange(5, N) if causal else np.arange(N)
        _close(out[:, rows], np.broadcast_to(vf[:, 5:6], (BH, rows.size, d)), 1e-20, "dominant key out")
        assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse)), "overflow with extreme scores"
        _close(lse[:, rows], np.full((BH, rows.size), 2048.0), 1e-12, "dominant key lse")
        out_r, lse_r = orc.ring(q, k, v, 4, causal, LAYOUT_STRIPED)
        _close(out_r, out, 1e-12, "dominant key ring")
        _close(lse_r, lse, 1e-12, "dominant key ring lse")


def pin_sdpa(orc):
    """Reduction to a library routine: torch's scaled_dot_product_attention in
    float64 on the CPU, and logsumexp of the masked score matrix."""
    for (BH, N, d) in ((2, 40, 16), (1, 33, 64), (3, 7, 1)):
        q, k, v = rand_bits((BH, N, d), 51 + N), rand_bits((BH, N, d), 52 + N), rand_bits((BH, N, d), 53 + N)
        qt, kt, vt = (torch.from_numpy(bits_to_f64(x)) for x in (q, k, v))
        for causal in (False, True):
            ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=causal)
            sc = torch.einsum("bqd,bkd->bqk", qt, kt) / math.sqrt(d)
            if causal:
                sc = sc.masked_fill(~torch.from_numpy(allowed_matrix(N, True)), float("-inf"))
            ref_lse = torch.logsumexp(sc, dim=-1)
            out, lse = orc.dense(q, k, v, causal)
            _close(out, ref.numpy(), 1e-12, "sdpa out")
            _close(lse, ref_lse.numpy(), 1e-12, "sdpa lse")


def band_matrix(N, window):
    """Causal sliding window: query t sees keys t-window+1 .. t."""
    t = np.arange(N)
    dist = t[:, None] - t[None, :]
    return (dist >= 0) & (dist < window)


def pin_window_closed_forms(orc):
    """Sliding window ([RA-CN] "正确性测试应覆盖哪些边界": sliding-window masks):
    window 1 leaves each query its own key only, so out_t = v_t and
    lse_t = s_tt exactly; a window of N or more is the plain causal mask."""
    BH, N, d = 2, 19, 8
    q, k, v = rand_bits((BH, N, d), 131), rand_bits((BH, N, d), 132), rand_bits((BH, N, d), 133)
    out, lse = orc.dense(q, k, v, True, window=1)
    qf, kf, vf = bits_to_f64(q), bits_to_f64(k), bits_to_f64(v)
    _close(out, vf, 0.0, "window 1 out = v")
    _close(lse, np.einsum("btd,btd->bt", qf, kf) / math.sqrt(d), 1e-13, "window 1 lse = own score")
    ref = orc.dense(q, k, v, True)
    for w in (N, N + 5):
        got = orc.dense(q, k, v, True, window=w)
        _close(got[0], ref[0], 0.0, f"window {w} = causal out")
        _close(got[1], ref[1], 0.0, f"window {w} = causal lse")


def pin_window_sdpa(orc):
    """Sliding window against torch's scaled_dot_product_attention in float64
    with the explicit band mask."""
    BH, N, d = 2, 37, 16
    q, k, v = rand_bits((BH, N, d), 141), rand_bits((BH, N, d), 142), rand_bits((BH, N, d), 143)
    qt, kt, vt = (torch.from_numpy(bits_to_f64(x)) for x in (q, k, v))
    for w in (2, 3, 8, 20):
        band = torch.from_numpy(band_matrix(N, w))
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=band)
        sc = (torch.einsum("bqd,bkd->bqk", qt, kt) / math.sqrt(d)).masked_fill(~band, float("-inf"))
        out, lse = orc.dense(q, k, v, True, window=w)
        _close(out, ref.numpy(), 1e-12, f"window {w} sdpa out")
        _close(lse, torch.logsumexp(sc, dim=-1).numpy(), 1e-12, f"window {w} sdpa lse")


# ------------------------------------------------------------------ the ring
def pin_ring_equals_dense(orc):
    """The ring reaches the dense result ([GRA] "Why partial results are
    allowed to merge": exact after P merges; [RA-CN] "局部 Softmax 为什么不能直接相加")
    for every divisor P of N, both layouts, causal and not."""
    for (BH, N, d) in ((2, 24, 4), (1, 16, 1), (1, 12, 64)):
        q, k, v = rand_bits((BH, N, d), 61 + d), rand_bits((BH, N, d), 62 + d), rand_bits((BH, N, d), 63 + d)
        for causal in (False, True):
            ref_out, ref_lse = orc.dense(q, k, v, causal)
            for P in [p for p in range(1, N + 1) if N % p == 0]:
                for layout in layouts_for(N, P):
                    out, lse = orc.ring(q, k, v, P, causal, layout)
                    tol = 1e-13 if P == 1 else 1e-12
                    _close(out, ref_out, tol, f"ring=dense out P={P} layout={layout} causal={causal}")
                    _close(lse, ref_lse, tol, f"ring=dense lse P={P} layout={layout} causal={causal}")


def pin_window_ring(orc):
    """With a sliding window the ring still reaches the dense result, in
    every layout, and visits exactly the pairs inside the band once."""
    BH, N, d = 1, 24, 4
    q, k, v = rand_bits((BH, N, d), 151), rand_bits((BH, N, d), 152), rand_bits((BH, N, d), 153)
    for w in (1, 2, 5, 13):
        ref_out, ref_lse = orc.dense(q, k, v, True, window=w)
        for P in (1, 2, 3, 4, 6):
            for layout in layouts_for(N, P):
                out, lse, cnt = orc.ring(q, k, v, P, True, layout, visits=True, window=w)
                _close(out, ref_out, 1e-12, f"window ring out w={w} P={P} layout={layout}")
                _close(lse, ref_lse, 1e-12, f"window ring lse w={w} P={P} layout={layout}")
                assert np.array_equal(cnt[0], band_matrix(N, w).astype(np.int64)), (w, P, layout)


def pin_layouts_agree(orc):
    """Contiguous, striped and zigzag layouts give the same natural-order
    result (a layout only changes which tokens each shard holds)."""
    BH, N, d = 2, 32, 8
    q, k, v = rand_bits((BH, N, d), 71), rand_bits((BH, N, d), 72), rand_bits((BH, N, d), 73)
    for causal in (False, True):
        for P in (2, 4, 8):
            a = orc.ring(q, k, v, P, causal, LAYOUT_CONTIGUOUS)
            for layout in (LAYOUT_STRIPED, LAYOUT_ZIGZAG):
                b = orc.ring(q, k, v, P, causal, layout)
                _close(a[0], b[0], 1e-12, f"layouts out {layout}")
                _close(a[1], b[1], 1e-12, f"layouts lse {layout}")


def pin_visits_exactly_once(orc):
    """Every allowed (q, k) pair is used exactly once and no other pair is
    ([RA-CN] "局部 Softmax 为什么不能直接相加": every allowed Q-K pair computed)."""
    BH, N, d = 1, 24, 2
    q, k, v = rand_bits((BH, N, d), 81), rand_bits((BH, N, d), 82), rand_bits((BH, N, d), 83)
    for causal in (False, True):
        want = allowed_matrix(N, causal).astype(np.int64)
        for P in (1, 2, 3, 4, 6, 8, 12, 24):
            for layout in layouts_for(N, P):
                _, _, cnt = orc.ring(q, k, v, P, causal, layout, visits=True)
                assert np.array_equal(cnt[0], want), f"visits P={P} layout={layout} causal={causal}"


def pin_shard_work_closed_forms(orc):
    """Allowed pairs per shard under the causal mask, from the visit counts:
    contiguous W_r = r n^2 + n(n+1)/2; striped W_r = (r+1) n(n+1)/2 +
    (P-1-r) n(n-1)/2; all sum to N(N+1)/2 ([GRA] "The causal mask wrecks the
    load balance": a linear ramp from one block of work to P).  Zigzag, with
    chunks of c = N/2P: the rows of chunks r and 2P-1-r see r c^2 + c(c+1)/2
    and (2P-1-r) c^2 + c(c+1)/2 pairs, W_r = 2P c^2 + c for every shard ([GRA]
    "Striping the sequence to flatten the triangle": the work is shared
    evenly)."""
    BH, N, d = 1, 24, 1
    q, k, v = rand_bits((BH, N, d), 91), rand_bits((BH, N, d), 92), rand_bits((BH, N, d), 93)
    for P in (2, 3, 4, 6):
        n = N // P
        for layout in layouts_for(N, P):
            _, _, cnt = orc.ring(q, k, v, P, True, layout, visits=True)
            per_row = cnt[0].sum(axis=1)
            for r in range(P):
                rows = [orc.position(layout, n, P, r, i) for i in range(n)]
                got = int(per_row[rows].sum())
                if layout == LAYOUT_CONTIGUOUS:
                    want = r * n * n + n * (n + 1) // 2
                elif layout == LAYOUT_STRIPED:
                    want = (r + 1) * n * (n + 1) // 2 + (P - 1 - r) * n * (n - 1) // 2
                else:
                    c = n // 2
                    want = 2 * P * c * c + c
                assert got == want, f"W_{r} layout={layout} P={P}: {got} != {want}"
            assert int(per_row.sum()) == N * (N + 1) // 2


def pin_naive_sum_differs(orc):
    """Summing per-block softmax outputs is wrong ([GRA] "Why partial results
    are allowed to merge"; [RA-CN] "局部 Softmax 为什么不能直接相加"): each block
    normalises to 1 on its own, so rows with two or more non-empty blocks
    differ from dense attention."""
    BH, N, d = 1, 16, 8
    q, k, v = rand_bits((BH, N, d), 101), rand_bits((BH, N, d), 102), rand_bits((BH, N, d), 103)
    for causal in (False, True):
        ref, _ = orc.dense(q, k, v, causal)
        naive = orc.naive_block_sum(q, k, v, 4, causal, LAYOUT_CONTIGUOUS)
        assert float(np.max(np.abs(naive - ref))) > 1e-2, "naive sum should differ"
        # with one block (P = 1) the naive sum is the dense result
        one = orc.naive_block_sum(q, k, v, 1, causal, LAYOUT_CONTIGUOUS)
        _close(one, ref, 1e-12, "naive sum with P=1")


def pin_merge_order_independent(orc):
    """The merge is associative and commutative: folding the P block partials
    of a shard in any order and bracketing gives the same state, and its
    finalize equals dense attention."""
    BH, N, d, P = 2, 32, 8, 4
    n = N // P
    q, k, v = rand_bits((BH, N, d), 111), rand_bits((BH, N, d), 112), rand_bits((BH, N, d), 113)
    rng = np.random.default_rng(5)
    for layout in layouts_for(N, P):
        for causal in (False, True):
            ref_out, ref_lse = orc.dense(q, k, v, causal)
            for r in range(P):
                pos = np.array([orc.position(layout, n, P, r, i) for i in range(n)])
                qs = np.ascontiguousarray(q[:, pos])
                parts = []
                for j in range(P):
                    kpos = np.array([orc.position(layout, n, P, j, i) for i in range(n)])
                    parts.append(orc.block_partial(qs, np.ascontiguousarray(k[:, kpos]),
                                                   np.ascontiguousarray(v[:, kpos]), P, causal, layout, r, j))
                results = []
                for trial in range(4):
                    order = rng.permutation(P)
                    if trial % 2 == 0:  # left fold
                        acc = [x.copy() for x in parts[order[0]]]
                        for j in order[1:]:
                            orc.merge_inplace(acc, parts[j])
                    else:  # pairwise tree
                        items = [[x.copy() for x in parts[j]] for j in order]
                        while len(items) > 1:
                            nxt = []
                            for a in range(0, len(items) - 1, 2):
                                orc.merge_inplace(items[a], items[a + 1])
                                nxt.append(items[a])
                            if len(items) % 2:
                                nxt.append(items[-1])
                            items = nxt
                        acc = items[0]
                    out, lse = orc.finalize(*acc)
                    results.append((out, lse))
                for out, lse in results:
                    _close(out, ref_out[:, pos], 1e-12, "merge order: out")
                    _close(lse, ref_lse[:, pos], 1e-12, "merge order: lse")


def pin_merge_empty_side(orc):
    """A side with m = -inf (a block with no allowed key) contributes nothing;
    two empty sides stay empty."""
    d = 3
    a = (np.array([0.5, -np.inf], np.float32), np.array([2.0, 0.0], np.float32),
         np.array([[1, 2, 3], [0, 0, 0]], np.float32))
    b = (np.array([-np.inf, -np.inf], np.float32), np.array([0.0, 0.0], np.float32), np.zeros((2, d), np.float32))
    m, l, o = orc.merge_states(a, b)
    assert m[0] == 0.5 and l[0] == 2.0 and np.array_equal(o[0], [1, 2, 3])
    assert m[1] == -np.inf and l[1] == 0.0 and np.array_equal(o[1], [0, 0, 0]) and not np.any(np.isnan(o))
    m2, l2, o2 = orc.merge_states(b, a)
    assert m2[0] == 0.5 and l2[0] == 2.0 and np.array_equal(o2[0], [1, 2, 3])


def pin_merge_two_point_example(orc):
    """Two one-key blocks with scores 0 and ln 4 in float32 states: the merged
    softmax weights are 1/5 and 4/5 (values chosen so the answer is known)."""
    ln4 = np.float32(math.log(4.0))
    a = (np.array([0.0], np.float32), np.array([1.0], np.float32), np.array([[10.0, 0.0]], np.float32))
    b = (np.array([ln4], np.float32), np.array([1.0], np.float32), np.array([[0.0, 5.0]], np.float32))
    m, l, o = orc.merge_states(a, b)
    out, lse = orc.finalize(m, l, o)
    w_b = 1.0 / (1.0 + math.exp(-float(ln4)))
    _close(out[0], [10.0 * (1 - w_b), 5.0 * w_b], 1e-15, "two-point merge out")
    _close(lse, [math.log(1.0 + math.exp(float(ln4)))], 1e-15, "two-point merge lse")
    assert abs(w_b - 0.8) < 1e-7


def pin_golden_schedule(orc):
    """The 4-device walk-through printed in [RA-CN] "环是怎样工作的": at step 0
    device r uses its own block; at step 1 device 0 holds block 3, device 1
    block 0, device 2 block 1, device 3 block 2."""
    path = os.path.join(GOLDEN, "ring_schedule_4dev.txt")
    rows = [ln.split() for ln in open(path) if ln.strip() and not ln.startswith("#")]
    assert rows
    for step, dev, blk in rows:
        assert orc.block_at(4, int(dev), int(step)) == int(blk), (step, dev, blk)


def pin_positions(orc):
    """Global positions: contiguous device p local i -> p*n + i ([RA-CN]
    "位置编码必须使用全局位置"); striped: token t on shard t mod P; zigzag
    ([GRA] "Striping the sequence to flatten the triangle"): shard 0 holds
    the very first and the very last chunk, the last shard the two middle
    chunks.  Every map is a bijection onto 0..N-1 and owner() inverts it."""
    n, P = 6, 4
    assert orc.position(LAYOUT_CONTIGUOUS, n, P, 2, 3) == 15
    assert orc.position(LAYOUT_STRIPED, n, P, 2, 3) == 14
    N, c = n * P, n // 2
    first, last = [orc.position(LAYOUT_ZIGZAG, n, P, 0, i) for i in range(n)], \
        [orc.position(LAYOUT_ZIGZAG, n, P, P - 1, i) for i in range(n)]
    assert first == list(range(c)) + list(range(N - c, N))
    assert last == list(range((P - 1) * c, (P + 1) * c))
    for layout in LAYOUTS:
        seen = sorted(orc.position(layout, n, P, r, i) for r in range(P) for i in range(n))
        assert seen == list(range(n * P))
        for r in range(P):
            for i in range(n):
                assert orc.owner(layout, n, P, orc.position(layout, n, P, r, i)) == (r, i)


# -------------------------------------------------------------- the backward
def _torch_grads(q, k, v, dout, mask):
    """float64 autograd of torch's scaled_dot_product_attention (a library
    routine) for the bf16 inputs widened exactly; mask is a boolean [N, N]
    (True = allowed) or None."""
    qt, kt, vt = (torch.from_numpy(bits_to_f64(x)).requires_grad_(True) for x in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(
        qt, kt, vt, attn_mask=None if mask is None else torch.from_numpy(mask))
    out.backward(torch.from_numpy(bits_to_f64(dout)))
    return qt.grad.numpy(), kt.grad.numpy(), vt.grad.numpy()


def _mask(N, causal, window=0):
    if window:
        return band_matrix(N, window)
    return allowed_matrix(N, True) if causal else None


def pin_bwd_autograd(orc):
    """Reduction to a library routine: the dense backward equals float64
    autograd through torch's scaled_dot_product_attention ([RA-CN] "Backward
    需要让梯度也沿环传播": every Q-K/V interaction contributes a gradient)."""
    for (BH, N, d, causal, w) in ((2, 19, 8, False, 0), (2, 24, 16, True, 0), (1, 33, 64, True, 0),
                                  (1, 21, 4, True, 5), (3, 5, 1, True, 0)):
        q, k, v, do = (rand_bits((BH, N, d), 300 + N + x) for x in range(4))
        ref = _torch_grads(q, k, v, do, _mask(N, causal, w))
        got = orc.dense_bwd(q, k, v, do, causal, window=w)
        for name, a, b in zip(("dq", "dk", "dv"), got, ref):
            _close(a, b, 1e-12, f"bwd autograd {name} N={N} d={d} causal={causal} w={w}")


def pin_bwd_finite_differences(orc):
    """Central differences of L = sum(dO * O), O from torch's float64
    scaled_dot_product_attention, at a few coordinates of q, k and v: an
    independent check of the chain rule (including the D = rowsum(dO * O)
    term of the softmax derivative)."""
    BH, N, d = 1, 10, 4
    q, k, v, do = (rand_bits((BH, N, d), 320 + x) for x in range(4))
    base = [torch.from_numpy(bits_to_f64(x)) for x in (q, k, v)]
    dof = torch.from_numpy(bits_to_f64(do))
    rng = np.random.default_rng(5)
    for causal in (False, True):
        grads = orc.dense_bwd(q, k, v, do, causal)
        for which in range(3):
            for _ in range(4):
                t, c = int(rng.integers(N)), int(rng.integers(d))
                h = 1e-5
                vals = []
                for sign in (1.0, -1.0):
                    xs = [b.clone() for b in base]
                    xs[which][0, t, c] += sign * h
                    o = torch.nn.functional.scaled_dot_product_attention(*xs, is_causal=causal)
                    vals.append(float((o * dof).sum()))
                fd = (vals[0] - vals[1]) / (2 * h)
                got = grads[which][0, t, c]
                assert abs(fd - got) <= 1e-7 * max(1.0, abs(got)), \
                    f"finite difference {'qkv'[which]}[{t},{c}] causal={causal}: {fd} vs {got}"


def pin_bwd_closed_forms(orc):
    """Closed forms: (a) every v row equal: O does not depend on q or k, so
    dq = dk = 0; (b) window 1 (each query sees only itself): P = 1, so dv = dO
    and dq = dk = 0; (c) N = 1: the same."""
    BH, N, d = 2, 12, 4
    q, k, do = rand_bits((BH, N, d), 331), rand_bits((BH, N, d), 332), rand_bits((BH, N, d), 333)
    c = np.array([0.75, -2.0, 0.125, 1.5], np.float32)
    v = to_bits(np.broadcast_to(c, (BH, N, d)))
    for causal in (False, True):
        dq, dk, _ = orc.dense_bwd(q, k, v, do, causal)
        _close(dq, 0.0, 1e-13, "constant v: dq")
        _close(dk, 0.0, 1e-13, "constant v: dk")
    v = rand_bits((BH, N, d), 334)
    dq, dk, dv = orc.dense_bwd(q, k, v, do, True, window=1)
    _close(dv, bits_to_f64(do), 0.0, "window 1: dv = dO")
    _close(dq, 0.0, 0.0, "window 1: dq")
    _close(dk, 0.0, 0.0, "window 1: dk")
    dq, dk, dv = orc.dense_bwd(q[:, :1], k[:, :1], v[:, :1], do[:, :1], False)
    _close(dv, bits_to_f64(do[:, :1]), 0.0, "N = 1: dv = dO")
    _close(dq, 0.0, 0.0, "N = 1: dq")


def pin_bwd_invariants(orc):
    """Identities of the gradients: each softmax row's dS sums to zero, so
    sum_k dK_k = 0; each probability row sums to one, so sum_k dV_k =
    sum_t dO_t; and sum_t q_t . dQ_t = sum_k k_k . dK_k (both are
    scale * sum dS_tk q_t . k_k), which a transposed dS would break."""
    BH, N, d = 2, 26, 8
    q, k, v, do = (rand_bits((BH, N, d), 340 + x) for x in range(4))
    qf, kf, dof = bits_to_f64(q), bits_to_f64(k), bits_to_f64(do)
    for causal, w in ((False, 0), (True, 0), (True, 7)):
        dq, dk, dv = orc.dense_bwd(q, k, v, do, causal, window=w)
        _close(dk.sum(1), 0.0, 1e-12, f"sum dK = 0 (causal={causal}, w={w})")
        _close(dv.sum(1), dof.sum(1), 1e-12, f"sum dV = sum dO (causal={causal}, w={w})")
        _close(np.einsum("btd,btd->b", qf, dq), np.einsum("btd,btd->b", kf, dk), 1e-12,
               f"q.dQ = k.dK (causal={causal}, w={w})")


def pin_bwd_rows_match(orc):
    """The sampled-row backward gives the same rows as the full one."""
    BH, N, d = 2, 30, 8
    q, k, v, do = (rand_bits((BH, N, d), 350 + x) for x in range(4))
    qrows, krows = [0, 7, 29, 13], [29, 0, 15, 28]
    for causal, w in ((False, 0), (True, 0), (True, 6)):
        full = orc.dense_bwd(q, k, v, do, causal, window=w)
        dq, dk, dv = orc.dense_bwd_rows(q, k, v, do, causal, qrows, krows, window=w)
        _close(dq, full[0][:, qrows], 1e-13, "rows dq")
        _close(dk, full[1][:, krows], 1e-13, "rows dk")
        _close(dv, full[2][:, krows], 1e-13, "rows dv")


def pin_bwd_keys_from_forward(orc):
    """dK and dV from the forward's saved out and lse (the oracle's dense
    forward) equal the full backward's at every key, causal or not, with a
    window and with packed documents."""
    BH, N, d = 2, 28, 8
    q, k, v, do = (rand_bits((BH, N, d), 370 + x) for x in range(4))
    keys = list(range(N))
    for causal, w, seg in ((False, 0, None), (True, 0, None), (True, 6, None), (True, 0, [0, 9, 10, 28])):
        full = orc.dense_bwd(q, k, v, do, causal, window=w, segments=seg)
        out, lse = orc.dense(q, k, v, causal, window=w, segments=seg)
        dk, dv = orc.dense_bwd_keys(q, k, v, do, out, lse, causal, keys, window=w, segments=seg)
        _close(dk, full[1], 1e-12, f"keys dk causal={causal} w={w} seg={seg}")
        _close(dv, full[2], 1e-12, f"keys dv causal={causal} w={w} seg={seg}")


def pin_ring_bwd_equals_dense(orc):
    """The ring backward (dQ kept by the query owner, dK and dV travelling
    with their block and returning to its owner; [RA-CN] "Backward
    需要让梯度也沿环传播") reaches the dense gradients for every divisor P of
    N, every layout, causal or not, with and without a window, and uses
    every allowed (query, key) pair exactly once."""
    for (BH, N, d) in ((2, 24, 4), (1, 12, 16)):
        q, k, v, do = (rand_bits((BH, N, d), 360 + d + x) for x in range(4))
        for causal, w in ((False, 0), (True, 0), (True, 5)):
            ref = orc.dense_bwd(q, k, v, do, causal, window=w)
            out, lse = orc.dense(q, k, v, causal, window=w)
            allowed = _mask(N, causal, w)
            allowed = np.ones((N, N), bool) if allowed is None else allowed
            for P in [p for p in range(1, N + 1) if N % p == 0]:
                for layout in layouts_for(N, P):
                    got = orc.ring_bwd(q, k, v, do, out, lse, P, causal, layout, visits=True, window=w)
                    for name, a, b in zip(("dq", "dk", "dv"), got[:3], ref):
                        _close(a, b, 1e-12, f"ring bwd {name} P={P} layout={layout} causal={causal} w={w}")
                    assert np.array_equal(got[3][0], allowed.astype(np.int64)), (P, layout, causal, w)


# ---------------------------------------------------------------- segments
def segment_matrix(bounds, N, causal, window=0):
    """Allowed (query, key) pairs of a packed sequence: same document, and
    the causal rule and window on top."""
    seg = np.repeat(np.arange(len(bounds) - 1), np.diff(bounds))
    m = seg[:, None] == seg[None, :]
    if causal or window:
        m &= _mask(N, True, window) if window else allowed_matrix(N, True)
    return m


def pin_segments_independent(orc):
    """Sequence packing ([RA-CN] "正确性测试应覆盖哪些边界": documents packed into
    one sequence must not attend to each other): the result on the packed
    sequence equals attention over each document on its own, and a valid
    length L (the tail padding as a document of its own) leaves the first L
    rows as attention over those L tokens alone."""
    BH, N, d = 2, 40, 8
    q, k, v = rand_bits((BH, N, d), 401), rand_bits((BH, N, d), 402), rand_bits((BH, N, d), 403)
    bounds = [0, 7, 20, 33, 40]
    for causal in (False, True):
        out, lse = orc.dense(q, k, v, causal, segments=bounds)
        for a, b in zip(bounds[:-1], bounds[1:]):
            sl = lambda x: np.ascontiguousarray(x[:, a:b])
            ref_o, ref_l = orc.dense(sl(q), sl(k), sl(v), causal)
            _close(out[:, a:b], ref_o, 1e-13, f"segment [{a},{b}) out causal={causal}")
            _close(lse[:, a:b], ref_l, 1e-13, f"segment [{a},{b}) lse causal={causal}")
        L = 29
        out, lse = orc.dense(q, k, v, causal, segments=[0, L, N])
        sl = lambda x: np.ascontiguousarray(x[:, :L])
        ref_o, ref_l = orc.dense(sl(q), sl(k), sl(v), causal)
        _close(out[:, :L], ref_o, 1e-13, f"valid length {L} out causal={causal}")
        _close(lse[:, :L], ref_l, 1e-13, f"valid length {L} lse causal={causal}")
    out1 = orc.dense(q, k, v, True, segments=[0, N])
    out0 = orc.dense(q, k, v, True)
    _close(out1[0], out0[0], 0.0, "one segment = no segments")


def pin_segments_sdpa(orc):
    """Segments against torch's float64 scaled_dot_product_attention with the
    explicit mask (same document, and causal / window)."""
    BH, N, d = 2, 37, 16
    q, k, v = rand_bits((BH, N, d), 411), rand_bits((BH, N, d), 412), rand_bits((BH, N, d), 413)
    qt, kt, vt = (torch.from_numpy(bits_to_f64(x)) for x in (q, k, v))
    bounds = [0, 5, 6, 19, 37]
    for causal, w in ((False, 0), (True, 0), (True, 6)):
        m = torch.from_numpy(segment_matrix(bounds, N, causal, w))
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=m)
        sc = (torch.einsum("bqd,bkd->bqk", qt, kt) / math.sqrt(d)).masked_fill(~m, float("-inf"))
        out, lse = orc.dense(q, k, v, causal, segments=bounds, window=w)
        _close(out, ref.numpy(), 1e-12, f"segments sdpa out causal={causal} w={w}")
        _close(lse, torch.logsumexp(sc, dim=-1).numpy(), 1e-12, f"segments sdpa lse causal={causal} w={w}")


def pin_segments_ring(orc):
    """With segments the ring reaches the dense result in every layout and
    uses exactly the allowed pairs once; the ring backward reaches the dense
    gradients, and those match float64 autograd through SDPA with the mask."""
    BH, N, d = 1, 24, 4
    q, k, v, do = (rand_bits((BH, N, d), 420 + x) for x in range(4))
    bounds = [0, 5, 13, 14, 24]
    for causal, w in ((False, 0), (True, 0), (True, 4)):
        ref_out, ref_lse = orc.dense(q, k, v, causal, segments=bounds, window=w)
        ref_g = orc.dense_bwd(q, k, v, do, causal, segments=bounds, window=w)
        auto = _torch_grads(q, k, v, do, segment_matrix(bounds, N, causal, w))
        for name, a, b in zip(("dq", "dk", "dv"), ref_g, auto):
            _close(a, b, 1e-12, f"segments bwd autograd {name} causal={causal} w={w}")
        allowed = segment_matrix(bounds, N, causal, w).astype(np.int64)
        for P in (1, 2, 3, 4, 6):
            for layout in layouts_for(N, P):
                out, lse, cnt = orc.ring(q, k, v, P, causal, layout, visits=True, segments=bounds, window=w)
                _close(out, ref_out, 1e-12, f"segments ring out P={P} layout={layout} causal={causal}")
                _close(lse, ref_lse, 1e-12, f"segments ring lse P={P} layout={layout} causal={causal}")
                assert np.array_equal(cnt[0], allowed), (P, layout, causal, w)
                g = orc.ring_bwd(q, k, v, do, ref_out, ref_lse, P, causal, layout, segments=bounds, window=w)
                for name, a, b in zip(("dq", "dk", "dv"), g, ref_g):
                    _close(a, b, 1e-12, f"segments ring bwd {name} P={P} layout={layout} causal={causal}")


ALL_PINS = [
    pin_equal_keys_closed_form,
    pin_constant_values,
    pin_causal_first_row,
    pin_dominant_key,
    pin_sdpa,
    pin_window_closed_forms,
    pin_window_sdpa,
    pin_ring_equals_dense,
    pin_window_ring,
    pin_layouts_agree,
    pin_visits_exactly_once,
    pin_shard_work_closed_forms,
    pin_naive_sum_differs,
    pin_merge_order_independent,
    pin_merge_empty_side,
    pin_merge_two_point_example,
    pin_golden_schedule,
    pin_positions,
    pin_bwd_autograd,
    pin_bwd_finite_differences,
    pin_bwd_closed_forms,
    pin_bwd_invariants,
    pin_bwd_rows_match,
    pin_bwd_keys_from_forward,
    pin_ring_bwd_equals_dense,
    pin_segments_independent,
    pin_segments_sdpa,
    pin_segments_ring,
]
