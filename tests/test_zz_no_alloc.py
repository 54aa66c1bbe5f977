"""ring_attn_fwd_noalloc: the ring forward for callers that cannot allocate
device memory (for example a plug-in inside a host application that owns all
device memory through its own pool, or a latency-critical path where
cudaMalloc/cudaFree may synchronise the device).  Its scratch lives in a
fixed array inside the library.

The GPU test calls it through the C ABI twice in a row and checks each
result against ring_attn_fwd (which takes a caller-allocated workspace),
within the parity tolerances of the other tests.  This file sorts last so a
run that stops at the first failure has already run every other test."""
import ctypes

import pytest
import torch

import ring_sequence_parallelism_gb300 as ra
from ring_sequence_parallelism_gb300 import _lib
from ring_sequence_parallelism_gb300.inputs import make_qkv

TOL_OUT = 1e-2
TOL_LSE = 1e-3


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


@pytest.mark.gpu
@pytest.mark.parametrize("layout", ["striped", "contiguous", "zigzag"])
def test_noalloc_matches_fwd_twice(lib, layout):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B, H, N, d, P = 1, 4, 4096, 128, 4
    q, k, v = (x.cuda() for x in make_qkv(B, H, N, d, seed=31))
    att = ra.RingAttention(B, H, N, d, P, causal=True, layout=layout)
    ref_out, ref_lse = att.fwd(q, k, v)
    att.check()
    stream = torch.cuda.current_stream().cuda_stream
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for call in range(2):
        out = torch.full((B, H, N, d), float("nan"), device="cuda")
        lse = torch.full((B, H, N), float("nan"), device="cuda")
        rc = lib.ring_attn_fwd_noalloc(att.handle, q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                       lse.data_ptr(), status.data_ptr(), stream)
        assert rc == 0, lib.ring_attn_last_error()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        d_out = float((out - ref_out).abs().max())
        d_lse = float((lse - ref_lse).abs().max())
        print(f"noalloc {layout} call {call}: max|dout|={d_out:.3e} max|dlse|={d_lse:.3e}")
        assert d_out <= TOL_OUT and d_lse <= TOL_LSE
    att.close()
