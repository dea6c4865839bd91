"""GPU: the bounded device-side waits give up instead of hanging.

Every streaming kernel waits on its mbarriers with the same bounded wait (0.5 s of
%globaltimer time once 1024 polls have been made, 2^21 polls at most). A wait that
runs out sets the timeout bit of the error word. The single-warp streaming kernel
then lets the warp's copies in flight land and returns; the tensor-core kernels,
whose warps meet at a CTA-wide barrier after every round, take the timed-out warp to
that barrier, and every warp leaves after it once its own copies have landed.

qmv_debug_wait_bound runs the wait in one thread on an mbarrier that nothing
completes; qmv_debug_cta_abort runs the multi-warp exit in a CTA of 8 warps, one of
which waits on copies that were never issued while the others consume real ones. No
fault and no trap: the waits themselves run out, the host reads the error status,
and the context stays usable.
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


def _context_usable(q):
    """A quantize call after the timeout matches the oracle byte for byte."""
    from gemm_qmv_quantize_gb300 import synth
    x = synth.activations_f32(2, 4096, seed=5, device="cuda")
    xq = q.qmv_quantize_q8_1(x)
    assert (xq.cpu().numpy() == oracle.quantize_q8_1(x.cpu().numpy())).all()
    assert q.error_flags() == 0


def test_wait_gives_up_flags_and_context_stays_usable(q):
    q.error_flags(clear=True)
    out = q.qmv_debug_wait_bound()
    torch.cuda.synchronize()
    done, ns = out.tolist()
    print(f"bounded wait gave up after {ns / 1e6:.3f} ms")
    assert done == 0
    assert 0.5e9 <= ns < 20e9      # the time bound, not the poll cap, ends it on a running GPU
    assert q.error_flags(clear=True) & 1
    assert q.error_flags() == 0
    _context_usable(q)


@pytest.mark.parametrize("stuck", [0, 3, 7])
def test_cta_leaves_together_after_one_warp_gives_up(q, stuck):
    q.error_flags(clear=True)
    out = q.qmv_debug_cta_abort(stuck)
    torch.cuda.synchronize()
    rec = out.cpu().tolist()
    print("per warp [gave up, saw abort, in flight, ns to barrier]:", rec)
    for w, (gave_up, saw_abort, inflight, ns) in enumerate(rec):
        # the abort word is set only when the stuck warp gives up (after its 0.5 s bound):
        # a warp that reads it set after the barrier has waited there for the stuck warp
        assert saw_abort == 1, f"warp {w} left the round without the stuck warp"
        if w == stuck:
            assert gave_up == 1 and inflight == 2    # both of its copies were never issued
            assert ns >= 0.5e9
        else:
            assert gave_up == 0 and inflight == 0    # its real copies landed and were consumed
    assert q.error_flags(clear=True) & 1
    _context_usable(q)
