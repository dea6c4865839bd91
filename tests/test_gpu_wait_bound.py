"""GPU: the bounded device-side wait gives up instead of hanging.

Every streaming kernel waits on its mbarriers with the same bounded wait; a wait
that runs out sets the timeout bit of the error word, lets the warp's own copies
land and returns. qmv_debug_wait_bound waits with that code on an mbarrier that
nothing completes (no fault, no trap: the wait itself runs out), so the test sees
the error status on the host and a usable context afterwards.
"""
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    from gemm_qmv_quantize_gb300 import build
    build.build()
    import gemm_qmv_quantize_gb300 as q
    return q


def test_wait_gives_up_flags_and_context_stays_usable(q):
    q.error_flags(clear=True)
    out = q.qmv_debug_wait_bound()
    torch.cuda.synchronize()
    done, ns = out.tolist()
    print(f"bounded wait gave up after {ns / 1e6:.3f} ms")
    assert done == 0
    assert 0 < ns < 10 * 10**9
    assert q.error_flags(clear=True) & 1
    assert q.error_flags() == 0
    # the context still works: a quantize call after the timeout matches the oracle byte for byte
    from gemm_qmv_quantize_gb300 import synth
    x = synth.activations_f32(2, 4096, seed=5, device="cuda")
    xq = q.qmv_quantize_q8_1(x)
    assert (xq.cpu().numpy() == oracle.quantize_q8_1(x.cpu().numpy())).all()
    assert q.error_flags() == 0
