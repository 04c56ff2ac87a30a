"""Failure detection on the GPU without a fault: a bounded device-side wait that runs out.

Every spin-wait in the library's kernels gives up after a wall-clock limit, records
MOE_ERR_TIMEOUT in a device error word and lets the kernel exit.  The self-test entry
point makes such a wait run out on purpose (an mbarrier that nothing arrives at, 2 ms
limit); the next moe_sync_check must report the timeout exactly once, and the context
must still run a full layer correctly afterwards.
"""

import pytest
import torch

import synth
from tests import helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import mixture_experts_layer_04_gb300 as m
    from mixture_experts_layer_04_gb300 import build

    build.build()
    m.load()
    return m


def test_bounded_wait_times_out_and_context_survives(moe):
    moe.sync_check()                                   # start from a clean error word
    done = torch.zeros(4, dtype=torch.int32, device="cuda")
    moe.debug_wait_timeout(2000, done)
    with pytest.raises(moe.MoEError) as ei:
        moe.sync_check()
    assert ei.value.status == 5                        # MOE_ERR_TIMEOUT
    assert int(done[0]) == 2                           # the wait gave up, it did not complete
    moe.sync_check()                                   # reported once, then cleared
    # the context is still usable: a layer runs and matches a second run bit for bit
    shape = synth.MoEShape("after_timeout", T=300, H=256, E=16, K=4, I=128, bias="normal")
    inp = synth.make_inputs(shape, device="cuda")
    a = H.LayerRun(moe, shape, inp)
    b = H.LayerRun(moe, shape, inp)
    a.run()
    b.run()
    moe.sync_check()
    assert torch.equal(a.y, b.y)
    assert torch.isfinite(a.y32).all()


def test_debug_wait_rejects_bad_arguments(moe):
    done = torch.zeros(4, dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoEError):
        moe.debug_wait_timeout(0, done)
    with pytest.raises(moe.MoEError):
        moe.debug_wait_timeout(2_000_000, done)
