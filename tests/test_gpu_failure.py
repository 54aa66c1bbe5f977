"""Failure detection on the GPU without a fault: every device-side wait is
bounded, so a wait that nothing completes ends with an error status the
host reads, and the context stays usable (GPU only)."""
import numpy as np
import pytest
import torch

import oracle
import ring_sequence_parallelism_gb300 as ra
from ring_sequence_parallelism_gb300.inputs import make_qkv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from ring_sequence_parallelism_gb300 import build

    build.build()
    ra._lib.load()


def test_wait_that_never_completes_reports_timeout_and_context_survives():
    B, H, N, d, P = 1, 1, 512, 128, 2  # 2 CTAs per step: the timeout costs ~2 x 20 ms
    q, k, v = (x.cuda() for x in make_qkv(B, H, N, d, seed=3))
    att = ra.RingAttention(B, H, N, d, P, causal=True, layout="striped")
    att.set_option(ra.RING_OPT_WAIT_LIMIT_NS, 20_000_000)  # 20 ms
    att.set_option(ra.RING_OPT_DEBUG_DROP_V_LOADS, 1)  # no V tile ever lands
    att.fwd(q, k, v)
    with pytest.raises(ra.RingAttnError) as e:
        att.check()
    assert e.value.status == ra._lib.RING_ERR_TIMEOUT
    # the error word was cleared and the context still works
    att.set_option(ra.RING_OPT_DEBUG_DROP_V_LOADS, 0)
    att.set_option(ra.RING_OPT_WAIT_LIMIT_NS, 2_000_000_000)
    out, lse = att.fwd(q, k, v)
    att.check()
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle.default().dense(q.reshape(B * H, N, d), k.reshape(B * H, N, d),
                                              v.reshape(B * H, N, d), True)
    assert np.max(np.abs(out.reshape(B * H, N, d).cpu().double().numpy() - ref_out)) <= 1e-2
    assert np.max(np.abs(lse.reshape(B * H, N).cpu().double().numpy() - ref_lse)) <= 1e-3
    att.close()
