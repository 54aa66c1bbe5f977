"""ring_attn_fwd_noalloc: the ring forward for callers that cannot allocate
device memory (for example a plug-in inside a host application that owns all
device memory through its own pool, or a latency-critical path where
cudaMalloc/cudaFree may synchronise the device).  Its scratch lives in a
fixed array inside the library.

The GPU tests call it through the C ABI twice in a row and check each result
against ring_attn_fwd (which takes a caller-allocated workspace) bit for bit:
both run the same step kernels on the same values in the same order; only
where the running state is kept between steps differs.  The shapes cover a
shard length that is not a whole number of 128-row tiles, grouped K/V
heads, a sliding window, a non-causal ring, and a handle whose first call is
the allocation-free one.  A last test makes a bounded wait run out (the
test hook that drops the V loads) and checks that the status output reports
it and that the next call clears it.  This file sorts last so a run that
stops at the first failure has already run every other test."""
import ctypes

import pytest
import torch

import ring_sequence_parallelism_gb300 as ra
from ring_sequence_parallelism_gb300 import _lib
from ring_sequence_parallelism_gb300.inputs import make_qkv


@pytest.fixture(scope="module")
def lib():
    from ring_sequence_parallelism_gb300 import build

    build.build()
    return _lib.load()


def test_noalloc_rejects_problems_above_its_fixed_scratch(lib):
    """Host-side size check (no GPU work happens before it): 16 heads x 128K
    tokens x d=128 needs about 1 GB of scratch, far above the 64 MiB array."""
    h = ctypes.c_void_p()
    assert lib.ring_attn_create(ctypes.byref(h), 1, 16, 131072, 128, 16, 1, 1) == 0
    fake = ctypes.c_void_p(1 << 20)  # aligned, never dereferenced: the size check comes first
    rc = lib.ring_attn_fwd_noalloc(h, fake, fake, fake, fake, fake, None, None)
    assert rc == _lib.RING_ERR_UNSUPPORTED
    assert b"scratch" in lib.ring_attn_last_error()
    assert lib.ring_attn_destroy(h) == 0


def test_noalloc_size_message_counts_kv_heads(lib):
    """With grouped K/V heads the packed K/V is smaller, so the largest
    problem the array takes is larger; the rejection message says so."""
    msgs = []
    for hkv in (16, 2):
        h = ctypes.c_void_p()
        assert lib.ring_attn_create_gqa(ctypes.byref(h), 1, 16, hkv, 1 << 20, 128, 16, 1, 1) == 0
        fake = ctypes.c_void_p(1 << 20)
        assert lib.ring_attn_fwd_noalloc(h, fake, fake, fake, fake, fake, None, None) == _lib.RING_ERR_UNSUPPORTED
        msgs.append(lib.ring_attn_last_error().decode())
        assert lib.ring_attn_destroy(h) == 0
    rows = [int(m.split("up to about ")[1].split()[0]) for m in msgs]
    assert rows[1] > 4 * rows[0], msgs


def noalloc(lib, att, q, k, v, status):
    B, H, N, d = q.shape
    out = torch.full((B, H, N, d), float("nan"), device="cuda")
    lse = torch.full((B, H, N), float("nan"), device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.ring_attn_fwd_noalloc(att.handle, q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                   lse.data_ptr(), status.data_ptr(), stream)
    assert rc == 0, lib.ring_attn_last_error()
    torch.cuda.synchronize()
    return out, lse


CASES = [
    # (B, H, Hkv, N, d, P, causal, layout, window, noalloc_first)
    (1, 4, 4, 4096, 128, 4, True, "striped", 0, False),
    (1, 4, 4, 4096, 128, 4, True, "contiguous", 0, False),
    (1, 4, 4, 4096, 128, 4, True, "zigzag", 0, False),
    (1, 2, 2, 4 * 1000, 128, 4, True, "striped", 0, True),  # n = 1000: a ragged last tile; fresh handle
    (2, 8, 2, 2048, 128, 4, True, "contiguous", 0, False),  # grouped K/V heads
    (1, 2, 2, 4 * 512, 64, 4, True, "striped", 700, False),  # sliding window
    (1, 2, 2, 3 * 256, 128, 3, False, "contiguous", 0, True),  # non-causal, odd P; fresh handle
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}kv{}N{}d{}P{}{}{}W{}{}".format(
    c[0], c[1], c[2], c[3], c[4], c[5], "c" if c[6] else "n", c[7][0], c[8], "-first" if c[9] else ""))
def test_noalloc_matches_fwd_twice(lib, case):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B, H, Hkv, N, d, P, causal, layout, window, first = case
    q, k, v = (x.cuda() for x in make_qkv(B, H, N, d, seed=31 + N + H, Hkv=Hkv))
    att = ra.RingAttention(B, H, N, d, P, causal=causal, layout=layout, kv_heads=Hkv)
    if window:
        att.set_option(ra.RING_OPT_WINDOW, window)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    got = []
    if first:  # the allocation-free call comes before any ring_attn_fwd on this handle
        got.append(noalloc(lib, att, q, k, v, status))
        assert int(status.item()) == 0
    ref_out, ref_lse = att.fwd(q, k, v)
    att.check()
    torch.cuda.synchronize()
    while len(got) < 2:
        got.append(noalloc(lib, att, q, k, v, status))
        assert int(status.item()) == 0
    for call, (out, lse) in enumerate(got):
        d_out = float((out - ref_out).abs().max())
        d_lse = float((lse - ref_lse).abs().max())
        print(f"noalloc {case} call {call}: max|dout|={d_out:.3e} max|dlse|={d_lse:.3e}")
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse), (call, d_out, d_lse)
    att.close()


@pytest.mark.gpu
def test_noalloc_reports_a_wait_that_runs_out(lib):
    """A bounded wait that nothing completes (the V loads dropped, 20 ms
    limit) ends the call with a nonzero status in the caller's device int;
    the next call clears the error word and matches ring_attn_fwd."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B, H, N, d, P = 1, 1, 512, 128, 2  # 2 CTAs per step: the timeout costs ~2 x 20 ms a step
    q, k, v = (x.cuda() for x in make_qkv(B, H, N, d, seed=3))
    att = ra.RingAttention(B, H, N, d, P, causal=True, layout="striped")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    att.set_option(ra.RING_OPT_WAIT_LIMIT_NS, 20_000_000)
    att.set_option(ra.RING_OPT_DEBUG_DROP_V_LOADS, 1)
    noalloc(lib, att, q, k, v, status)
    assert int(status.item()) != 0
    att.set_option(ra.RING_OPT_DEBUG_DROP_V_LOADS, 0)
    att.set_option(ra.RING_OPT_WAIT_LIMIT_NS, 2_000_000_000)
    out, lse = noalloc(lib, att, q, k, v, status)
    assert int(status.item()) == 0
    ref_out, ref_lse = att.fwd(q, k, v)
    att.check()
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
    att.close()
