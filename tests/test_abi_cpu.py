"""C-ABI library on the CPU: it loads, exports every declared symbol, checks
its arguments, and its host planner matches the closed forms and the
oracle's visit counts.  No compute call is made (no GPU here)."""
import ctypes
import os
import re

import numpy as np
import pytest

import ring_sequence_parallelism_gb300 as ra
from ring_sequence_parallelism_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ringattn.h")


@pytest.fixture(scope="module")
def lib():
    from ring_sequence_parallelism_gb300 import build

    build.build()
    return _lib.load()


def declared_symbols():
    text = open(HEADER, encoding="utf-8").read()
    return sorted(set(re.findall(r"RINGATTN_API\s+(?:const\s+)?\w+\*?\s+\*?(ring_attn_\w+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_symbols()
    for must in ("ring_attn_create", "ring_attn_block_partial", "ring_attn_merge", "ring_attn_fwd",
                 "ring_attn_destroy"):
        assert must in names
    assert set(names) == set(_lib.SIGNATURES), "binding and header disagree"


def test_header_compiles_as_plain_c():
    """include/ringattn.h is a C header: plain C99 with warnings on, no C++
    or CUDA types in the signatures."""
    import shutil
    import subprocess

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    r = subprocess.run([cc, "-x", "c", "-std=c99", "-fsyntax-only", "-Wall", "-Wextra", "-Werror", HEADER],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_c_program_against_the_library(lib, tmp_path):
    """tests/c_abi_host.c, a plain C program, built against the header and
    linked with libringattn.so, runs the host-side calls (no GPU needed)."""
    import shutil
    import subprocess

    from ring_sequence_parallelism_gb300 import build

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    libdir = os.path.dirname(build.LIBRARY)
    exe = str(tmp_path / "c_abi_host")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                        os.path.join(ROOT, "tests", "c_abi_host.c"), "-o", exe, "-L", libdir, "-lringattn",
                        "-Wl,-rpath," + libdir], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr


def test_library_exports_every_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def _create(lib, *args):
    h = ctypes.c_void_p()
    rc = lib.ring_attn_create(ctypes.byref(h), *args)
    return rc, h


@pytest.mark.parametrize("args,status", [
    ((0, 1, 64, 64, 1, 0, 0), _lib.RING_ERR_INVALID_ARG),      # B = 0
    ((1, 1, 64, 64, 0, 0, 0), _lib.RING_ERR_INVALID_ARG),      # P = 0
    ((1, 1, 64, 64, 1, 2, 0), _lib.RING_ERR_INVALID_ARG),      # causal = 2
    ((1, 1, 64, 64, 1, 0, 7), _lib.RING_ERR_INVALID_ARG),      # bad layout
    ((1, 1, 4, 64, 8, 0, 0), _lib.RING_ERR_INVALID_ARG),       # P > N
    ((1, 1, 100, 64, 3, 0, 0), _lib.RING_ERR_UNSUPPORTED),     # N % P != 0
    ((1, 1, 128, 96, 1, 0, 0), _lib.RING_ERR_UNSUPPORTED),     # d = 96
    ((1, 1, 4096, 64, 2048, 0, 0), _lib.RING_ERR_UNSUPPORTED),  # P above the table size
])
def test_create_rejects(lib, args, status):
    rc, h = _create(lib, *args)
    assert rc == status
    assert h.value is None
    assert lib.ring_attn_last_error()


def test_create_null_out(lib):
    assert lib.ring_attn_create(None, 1, 1, 64, 64, 1, 0, 0) == _lib.RING_ERR_INVALID_ARG


def test_calls_reject_null_arguments_without_a_gpu(lib):
    rc, h = _create(lib, 1, 2, 256, 64, 2, 1, 1)
    assert rc == 0
    st = _lib.RingState(None, None, None)
    assert lib.ring_attn_merge(h, st, st, None) == _lib.RING_ERR_INVALID_ARG
    assert lib.ring_attn_fwd(h, None, None, None, None, None, None, None) == _lib.RING_ERR_INVALID_ARG
    assert lib.ring_attn_block_partial(h, 0, 0, None, None, None, st, 0, None) == _lib.RING_ERR_INVALID_ARG
    assert lib.ring_attn_fwd_host(h, None, None, None, None, None, None) == _lib.RING_ERR_INVALID_ARG
    assert lib.ring_attn_set_option(h, 99, 1) == _lib.RING_ERR_INVALID_ARG
    for mode in (0, 1, 2):
        assert lib.ring_attn_set_option(h, _lib.RING_OPT_ROTATION, mode) == 0
    assert lib.ring_attn_set_option(h, _lib.RING_OPT_ROTATION, 3) == _lib.RING_ERR_INVALID_ARG
    assert lib.ring_attn_get_timing(h, None, None, None, None) == _lib.RING_ERR_INVALID_ARG
    assert lib.ring_attn_plan_block(h, 2, 0, None, None, None) == _lib.RING_ERR_INVALID_ARG
    assert lib.ring_attn_destroy(h) == 0
    assert lib.ring_attn_destroy(None) == 0


def test_workspace_size(lib):
    # rotation buffers (2 x K and V, bf16) + the running state in 128-row
    # tiles per shard: O~ (d floats) and m, l per row
    att = ra.RingAttention(1, 16, 131072, 128, 16, causal=True, layout="striped")
    elems = 16 * 131072 * 128
    assert att.workspace_size() == 4 * elems * 2 + 16 * 131072 * (128 + 2) * 4
    att.close()
    # ragged shards round up to whole tiles: n = 200 -> 2 tiles of 128 rows
    att = ra.RingAttention(2, 2, 3 * 200, 64, 3, causal=True, layout="contiguous")
    rows = 2 * 2 * 3 * 256
    up = lambda x: (x + 255) // 256 * 256
    assert att.workspace_size() == 4 * (2 * 2 * 600 * 64) * 2 + up(rows * 64 * 4) + 2 * up(rows * 4)
    att.close()


def test_fwd_host_checks_its_arguments(lib):
    """RingAttention.fwd_host rejects tensors of the wrong place, dtype or
    shape before any device work (host bf16 q, k, v; host fp32 out, lse)."""
    import torch

    att = ra.RingAttention(1, 2, 256, 64, 2, causal=True, layout="striped")
    q = torch.zeros(1, 2, 256, 64, dtype=torch.bfloat16)
    bad = [
        (q.float(), q, q, None, None),  # q not bf16
        (q, q[:, :1].contiguous(), q, None, None),  # k of the wrong shape
        (q, q, q.transpose(2, 3), None, None),  # v not contiguous
        (q, q, q, torch.zeros(1, 2, 256, 64, dtype=torch.bfloat16), None),  # out not fp32
        (q, q, q, None, torch.zeros(1, 2, 255)),  # lse of the wrong shape
    ]
    for args in bad:
        with pytest.raises(ValueError):
            att.fwd_host(*args)
    att.close()


def test_bwd_workspace_size_follows_the_schedule(lib):
    """The backward's workspace: -lse log2(e) and -D per row (shard-major,
    rows padded to whole tiles), plus, for one launch per ring step only,
    two buffers each of the travelling dK~ and dV~ (fp32, K/V heads)."""
    up = lambda x: (x + 255) // 256 * 256
    B, H, Hkv, N, d, P = 1, 8, 2, 4096, 128, 4
    att = ra.RingAttention(B, H, N, d, P, causal=True, layout="striped", kv_heads=Hkv)
    vec = up(B * H * P * 1024 * 4)  # n = 1024: 8 tiles of 128 rows
    acc = up(B * Hkv * N * d * 4)
    assert att.bwd_workspace_size() == 2 * vec  # lap schedule (the default)
    att.set_option(ra.RING_OPT_BWD_LAP, 0)
    assert att.bwd_workspace_size() == 2 * vec + 4 * acc
    att.set_option(ra.RING_OPT_BWD_LAP, 1)
    assert att.bwd_workspace_size() == 2 * vec
    for bad in (2, -1):
        assert lib.ring_attn_set_option(att.handle, _lib.RING_OPT_BWD_LAP, bad) == _lib.RING_ERR_INVALID_ARG
    att.close()
    # one shard: a single step, which needs no accumulator buffers either way
    att = ra.RingAttention(1, 2, 512, 64, 1, causal=True, layout="contiguous")
    att.set_option(ra.RING_OPT_BWD_LAP, 0)
    assert att.bwd_workspace_size() == 2 * up(2 * 1 * 512 * 4)
    att.close()


# -------------------------------------------------------------- planner
def test_plan_matches_golden_schedule(lib):
    """The 4-device walk-through in "Ring Attention：把超长序列沿设备环流动",
    section "环是怎样工作的"."""
    path = os.path.join(ROOT, "tests", "golden", "ring_schedule_4dev.txt")
    att = ra.RingAttention(1, 1, 4 * 128, 64, 4, causal=False, layout="contiguous")
    for line in open(path):
        if line.strip() and not line.startswith("#"):
            step, dev, blk = map(int, line.split())
            assert att.plan_block(dev, step)[0] == blk
    att.close()


@pytest.mark.parametrize("layout", ["contiguous", "striped"])
@pytest.mark.parametrize("P,n", [(2, 128), (4, 200), (8, 1024), (16, 8192), (64, 16384), (3, 1)])
def test_shard_work_closed_forms(lib, layout, P, n):
    """Allowed pairs per shard under the causal mask: contiguous
    W_r = r n^2 + n(n+1)/2, striped W_r = (r+1) n(n+1)/2 + (P-1-r) n(n-1)/2;
    the total is N(N+1)/2 ("GPU Ring Attention", "The causal mask wrecks the
    load balance": work ramps from one block on rank 0 to P on the last)."""
    B, H = 1, 2
    N = P * n
    att = ra.RingAttention(B, H, N, 64, P, causal=True, layout=layout)
    pairs, tiles = att.shard_work()
    for r in range(P):
        if layout == "contiguous":
            want = r * n * n + n * (n + 1) // 2
        else:
            want = (r + 1) * n * (n + 1) // 2 + (P - 1 - r) * n * (n - 1) // 2
        assert pairs[r] == want * B * H, (r, pairs[r], want)
    assert sum(pairs) == B * H * N * (N + 1) // 2
    steps = [att.step_work(s)[0] for s in range(P)]
    assert sum(steps) == sum(pairs)
    # every computed 128x128 tile covers at least one allowed pair
    assert sum(tiles) * 128 * 128 >= sum(pairs)
    if P > 1 and n >= 128:
        ratio = max(pairs) / min(pairs)
        if layout == "contiguous":
            assert ratio > P  # ~ 2P - 1
        else:
            assert ratio < 1.02
    att.close()


@pytest.mark.parametrize("layout", ["contiguous", "striped"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("P", [1, 2, 3, 6])
def test_planner_agrees_with_oracle_visits(lib, orc, layout, causal, P):
    """Per (shard, step) allowed-pair counts from the planner equal the
    oracle ring simulation's visit counts."""
    from oracle import LAYOUT_CONTIGUOUS, LAYOUT_STRIPED
    import oracle_pins

    N, d = 24, 2
    n = N // P
    lid = LAYOUT_STRIPED if layout == "striped" else LAYOUT_CONTIGUOUS
    q = oracle_pins.rand_bits((1, N, d), 1)
    _, _, cnt = orc.ring(q, q, q, P, causal, lid, visits=True)
    att = ra.RingAttention(1, 1, N, 64, P, causal=causal, layout=layout)
    for r in range(P):
        rows = [orc.position(lid, n, P, r, i) for i in range(n)]
        for s in range(P):
            j, cls, delta = att.plan_block(r, s)
            assert j == orc.block_at(P, r, s)
            cols = [orc.position(lid, n, P, j, kk) for kk in range(n)]
            got = int(cnt[0][np.ix_(rows, cols)].sum())
            # the planner's (class, delta) rule, enumerated
            want = sum(1 for i in range(n) for kk in range(n) if cls != 0 and kk - i <= delta)
            assert got == want, (r, s, j, cls, delta, got, want)
            if cls == 0:
                assert got == 0
            if cls == 1:
                assert got == n * n
    att.close()


@pytest.mark.parametrize("P,n", [(1, 256), (2, 256), (4, 512), (16, 8192), (64, 16384)])
def test_zigzag_shard_work_is_balanced(lib, P, n):
    """Zigzag ("GPU Ring Attention", "Striping the sequence to flatten the
    triangle"): every shard holds one early and one late chunk of c = n/2
    tokens and does the same causal work, W_r = 2P c^2 + c."""
    B, H, c = 1, 2, n // 2
    att = ra.RingAttention(B, H, P * n, 64, P, causal=True, layout="zigzag")
    pairs, tiles = att.shard_work()
    assert pairs == [(2 * P * c * c + c) * B * H] * P
    assert sum(pairs) == B * H * (P * n) * (P * n + 1) // 2
    assert sum(att.step_work(s)[0] for s in range(P)) == sum(pairs)
    assert sum(tiles) * 128 * 128 >= sum(pairs)
    att.close()


@pytest.mark.parametrize("P", [1, 2, 3])
@pytest.mark.parametrize("causal", [False, True])
def test_zigzag_plan_agrees_with_oracle(lib, orc, P, causal):
    """The planner's per-row mask (ring_attn_plan_mask: k < key_limit and
    k - row <= delta) admits exactly the keys the oracle's global positions
    allow, for every shard, step and row; per-block counts equal the oracle
    ring simulation's visits."""
    from oracle import LAYOUT_ZIGZAG
    import oracle_pins

    n = 256
    N, d = P * n, 2
    q = oracle_pins.rand_bits((1, N, d), 3)
    _, _, cnt = orc.ring(q, q, q, P, causal, LAYOUT_ZIGZAG, visits=True)
    att = ra.RingAttention(1, 1, N, 64, P, causal=causal, layout="zigzag")
    for r in range(P):
        qpos = np.array([orc.position(LAYOUT_ZIGZAG, n, P, r, i) for i in range(n)])
        for s in range(P):
            j, cls, _ = att.plan_block(r, s)
            assert j == orc.block_at(P, r, s)
            kpos = np.array([orc.position(LAYOUT_ZIGZAG, n, P, j, k) for k in range(n)])
            ks = np.arange(n)
            total = 0
            for i in range(n):
                klim, delta = att.plan_mask(r, s, i)
                rule = (ks < klim) & (ks - i <= delta)
                want = (kpos <= qpos[i]) if causal else np.ones(n, bool)
                assert np.array_equal(rule, want), (r, s, i)
                total += int(rule.sum())
            assert total == int(cnt[0][np.ix_(qpos, kpos)].sum())
            assert cls == (ra.RING_BLOCK_FULL if total == n * n else
                           ra.RING_BLOCK_DIAG if j == r else ra.RING_BLOCK_PARTIAL), (r, s, cls)
    att.close()


@pytest.mark.parametrize("P,n,causal,window,bounds", [
    (2, 256, True, 100, None), (3, 256, True, 300, None), (4, 512, True, 700, None), (2, 256, True, 1, None),
    (3, 256, True, 0, [0, 100, 101, 500, 768]), (2, 256, False, 0, [0, 300, 512]),
    (4, 256, True, 200, [0, 5, 600, 1024]),
])
def test_zigzag_window_and_segments_plan(lib, orc, P, n, causal, window, bounds):
    """Zigzag with a sliding window or documents: every row's key range
    (ring_attn_plan_key_range) is exactly the set of keys the oracle's ring
    simulation visits for it (one interval in the block's local order), the
    per-shard and per-step pair counts add up to the oracle's, and a block
    with no allowed pair is SKIP."""
    from oracle import LAYOUT_ZIGZAG
    import oracle_pins

    N, d = P * n, 2
    q = oracle_pins.rand_bits((1, N, d), 5)
    _, _, cnt = orc.ring(q, q, q, P, causal, LAYOUT_ZIGZAG, visits=True, window=window, segments=bounds)
    att = ra.RingAttention(1, 1, N, 64, P, causal=causal, layout="zigzag")
    if window:
        att.set_option(ra.RING_OPT_WINDOW, window)
    if bounds is not None:
        att.set_segments(bounds)
    pairs, _ = att.shard_work()
    assert sum(pairs) == int(cnt[0].sum())
    for r in range(P):
        qpos = np.array([orc.position(LAYOUT_ZIGZAG, n, P, r, i) for i in range(n)])
        shard_total = 0
        for s in range(P):
            j, cls, _ = att.plan_block(r, s)
            kpos = np.array([orc.position(LAYOUT_ZIGZAG, n, P, j, k) for k in range(n)])
            block_total = 0
            for i in range(n):
                first, last = att.plan_key_range(r, s, i)
                visited = np.nonzero(cnt[0][qpos[i], kpos])[0]
                want = np.arange(first, last + 1) if first <= last else np.array([], dtype=np.int64)
                assert np.array_equal(visited, want), (r, s, i, first, last, visited[:5])
                block_total += visited.size
            assert (cls == ra.RING_BLOCK_SKIP) == (block_total == 0), (r, s, cls, block_total)
            shard_total += block_total
        assert shard_total == pairs[r], (r, shard_total, pairs[r])
    att.close()


def test_grouped_query_handles(lib):
    """ring_attn_create_gqa: H must be a positive multiple of Hkv; the
    workspace holds the rotation buffers of the Hkv heads only."""
    h = ctypes.c_void_p()
    assert lib.ring_attn_create_gqa(ctypes.byref(h), 1, 6, 4, 1024, 64, 4, 1, 1) == _lib.RING_ERR_INVALID_ARG
    assert lib.ring_attn_create_gqa(ctypes.byref(h), 1, 6, 0, 1024, 64, 4, 1, 1) == _lib.RING_ERR_INVALID_ARG
    full = ra.RingAttention(1, 16, 131072, 128, 16, causal=True, layout="striped")
    gqa = ra.RingAttention(1, 16, 131072, 128, 16, causal=True, layout="striped", kv_heads=4)
    per_head = 131072 * 128 * 2  # one K or V buffer of one head, bf16
    assert full.workspace_size() - gqa.workspace_size() == 4 * (16 - 4) * per_head  # X and Y, K and V
    full.close()
    gqa.close()


def test_zigzag_needs_whole_tile_chunks(lib):
    """Chunks of N/2P tokens must be multiples of the 128-row tile."""
    h = ctypes.c_void_p()
    assert lib.ring_attn_create(ctypes.byref(h), 1, 1, 4 * 200, 64, 2, 1, ra.RING_LAYOUT_ZIGZAG) == \
        _lib.RING_ERR_UNSUPPORTED
    assert b"zigzag" in lib.ring_attn_last_error()
    assert lib.ring_attn_create(ctypes.byref(h), 1, 1, 4 * 256, 64, 2, 1, ra.RING_LAYOUT_ZIGZAG) == 0
    assert lib.ring_attn_destroy(h) == 0


def test_step_time_model_golden():
    """Pipelined ring time P x max(T_compute, T_comm): the worked estimate in
    "Ring Attention：把超长序列沿设备环流动", section "一个容量与时间的估算示例"."""
    from ring_sequence_parallelism_gb300.report import pipelined_ring_ms

    path = os.path.join(ROOT, "tests", "golden", "step_time_estimate.txt")
    for line in open(path):
        if line.strip() and not line.startswith("#"):
            steps, tc, tm, total = map(float, line.split())
            assert pipelined_ring_ms(int(steps), tc, tm) == pytest.approx(total)


@pytest.mark.parametrize("layout", ["contiguous", "striped"])
@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 5)])
@pytest.mark.parametrize("P", [1, 2, 3, 4])
def test_segment_plan_agrees_with_oracle(lib, orc, layout, causal, window, P):
    """With sequence packing the planner's key range of every (shard, step,
    row) and its per-step pair counts equal the pairs the oracle's ring
    simulation visits (same documents, causal rule and window)."""
    from oracle import LAYOUT_CONTIGUOUS, LAYOUT_STRIPED
    import oracle_pins

    N, d = 24, 2
    n = N // P
    bounds = [0, 5, 13, 14, 24]
    lid = LAYOUT_STRIPED if layout == "striped" else LAYOUT_CONTIGUOUS
    q = oracle_pins.rand_bits((1, N, d), 3)
    _, _, cnt = orc.ring(q, q, q, P, causal, lid, visits=True, window=window, segments=bounds)
    att = ra.RingAttention(1, 1, N, 64, P, causal=causal, layout=layout)
    if window:
        att.set_option(ra.RING_OPT_WINDOW, window)
    att.set_segments(bounds)
    for s in range(P):
        step_pairs = 0
        for r in range(P):
            j = orc.block_at(P, r, s)
            for i in range(n):
                tq = orc.position(lid, n, P, r, i)
                first, last = att.plan_key_range(r, s, i)
                want = [kk for kk in range(n) if cnt[0][tq, orc.position(lid, n, P, j, kk)]]
                got = list(range(max(first, 0), min(last, n - 1) + 1))
                assert got == want, (r, s, i, first, last, want)
                step_pairs += len(want)
        assert att.step_work(s)[0] == step_pairs, (s, att.step_work(s), step_pairs)
    att.set_segments(None)
    att.close()


def test_segments_rejected(lib):
    """Boundaries must rise strictly from 0 to N; the handle keeps its
    previous segments on an error."""
    att = ra.RingAttention(1, 1, 64, 64, 4, causal=True, layout="striped")
    for bad in ([0, 10, 10, 64], [1, 64], [0, 63], [0, 70, 64]):
        with pytest.raises(_lib.RingAttnError) as e:
            att.set_segments(bad)
        assert e.value.status == _lib.RING_ERR_INVALID_ARG
    att.close()
