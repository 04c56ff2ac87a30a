"""Failure detection on the GPU without a fault: a bounded device-side wait that runs out,
host-side injected faults, and the bounds-checking debug build.

Every spin-wait in the library's kernels gives up after a wall-clock limit, records
MOE_ERR_TIMEOUT in a device error word and lets the kernel exit.  The self-test entry
point makes such a wait run out on purpose (an mbarrier that nothing arrives at, 2 ms
limit); the next moe_sync_check must report the timeout exactly once, and the context
must still run a full layer correctly afterwards.
"""

import ctypes

import numpy as np
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


# ---------------------------------------------------------------- fault injection ----
# A fault injected inside moe_layer_forward (moe_debug_set_fault) makes the call fail after
# its earlier stages were enqueued, as a failed launch would.  The caller's output y must
# be untouched, the stream and the device must stay usable, and the next call must give
# exactly what an undisturbed call gives.  (Page "MoE大模型的智能调度…" §3.2 recounts
# production failures of the routing step; this rehearses a caller's clean-up on the host.)

@pytest.mark.parametrize("point", ["moe_layer_forward.route", "moe_layer_forward.permute",
                                   "moe_layer_forward.gate_up", "moe_layer_forward.shared",
                                   "moe_layer_forward.down", "moe_layer_forward.combine"])
@pytest.mark.parametrize("fused", [False, True], ids=["gather_combine", "fused_combine"])
@pytest.mark.parametrize("T", [700, 1100])   # from 1024 tokens the shared expert runs on a side stream
def test_injected_fault_leaves_output_untouched(moe, point, fused, T):
    shape = synth.MoEShape("fault", T=T, H=256, E=32, K=4, I=128, I_shared=64, theta=0.05,
                           bias="zipf", seed=13)
    inp = synth.make_inputs(shape, device="cuda")
    flags = moe.FLAG_FUSED_COMBINE if fused else 0
    clean = H.LayerRun(moe, shape, inp, flags=flags)
    clean.run()
    run = H.LayerRun(moe, shape, inp, flags=flags)
    run.y.fill_(7.0)
    moe.debug_set_fault(point, 1)
    try:
        with pytest.raises(moe.MoEError) as ei:
            run.run()
    finally:
        moe.debug_set_fault(None)
    assert ei.value.status == 4                        # MOE_ERR_CUDA, as a failed launch
    moe.sync_check()                                   # nothing went wrong on the device
    assert bool((run.y == 7.0).all()), "y was written by a call that failed"
    run.run()                                          # the next call runs normally
    moe.sync_check()
    if fused:   # the fused combine adds in no fixed order
        torch.testing.assert_close(run.y32, clean.y32, rtol=1e-5, atol=1e-5)
    else:
        assert torch.equal(run.y, clean.y) and torch.equal(run.y32, clean.y32)


# ---------------------------------------------------------------- debug build ----
# The bounds-checking build (-DMOE_DEBUG): on valid inputs it reports nothing and computes
# what the normal build computes; given an index out of range (which the normal build
# trusts), its kernel skips that access and moe_sync_check reports MOE_ERR_INTERNAL.  Each
# bad index below is compared against its bound before anything is read through it.

@pytest.fixture(scope="module")
def dbg(moe):
    from mixture_experts_layer_04_gb300 import build

    build.build(debug=True)
    return moe.load_debug()


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _s():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("fused", [False, True], ids=["gather_combine", "fused_combine"])
def test_debug_build_on_valid_inputs_reports_nothing(moe, dbg, fused):
    shape = synth.MoEShape("dbg_ok", T=600, H=512, E=64, K=8, I=256, I_shared=128, theta=0.05,
                           bias="zipf", seed=14)
    inp = synth.make_inputs(shape, device="cuda")
    flags = moe.FLAG_FUSED_COMBINE if fused else 0
    rel = H.LayerRun(moe, shape, inp, flags=flags)
    rel.run()
    moe.sync_check()
    d = H.LayerRun(moe, shape, inp, flags=flags)
    i = inp
    st = dbg.moe_layer_forward(ctypes.byref(d.cfg), _p(i["x"]), _p(i["w_router"]),
                               _p(i["router_bias"]), _p(i["w_gate_up"]), _p(i["w_down"]),
                               _p(i["w_shared_gate_up"]), _p(i["w_shared_down"]), _p(d.y),
                               _p(d.y32), _p(d.ws), ctypes.c_size_t(d.ws.numel()), _s())
    assert st == 0
    assert dbg.moe_sync_check(_s()) == 0
    torch.testing.assert_close(d.y32, rel.y32, rtol=1e-5, atol=1e-5)
    r_dbg, r_rel = d.routing(), rel.routing()
    for k in ("ids", "counts", "offsets", "inv"):
        np.testing.assert_array_equal(r_dbg[k], r_rel[k])


def test_debug_build_reports_out_of_range_inverse_map(dbg):
    import mixture_experts_layer_04_gb300 as m

    T, Hd, K = 300, 256, 4
    cfg = m.MoEConfig.make(T, Hd, 16, K, 128, 0, 0.0, m.BF16)
    g = torch.Generator(device="cuda").manual_seed(3)
    out_perm = torch.randn(T * K, Hd, device="cuda", generator=g)
    w = torch.full((T * K,), 0.25, device="cuda")
    inv = torch.arange(T * K, dtype=torch.int32, device="cuda")
    inv[7] = T * K + 1000                   # token 1, slot 3: past the last row
    y = torch.empty(T, Hd, dtype=torch.bfloat16, device="cuda")
    y32 = torch.empty(T, Hd, device="cuda")
    assert dbg.moe_combine(ctypes.byref(cfg), _p(out_perm), _p(inv), _p(w), None, _p(y),
                           _p(y32), _s()) == 0
    assert dbg.moe_sync_check(_s()) == 6    # MOE_ERR_INTERNAL
    assert dbg.moe_sync_check(_s()) == 0    # reported once
    ref = (out_perm.view(T, K, Hd) * 0.25).sum(1)
    ref[1] -= 0.25 * out_perm[7]            # the bad slot was skipped
    torch.testing.assert_close(y32, ref, rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("T", [100, 700])   # the one-launch and the three-launch permutation
def test_debug_build_reports_out_of_range_expert_id(dbg, T):
    import mixture_experts_layer_04_gb300 as m

    E, K, Hd = 16, 4, 128
    cfg = m.MoEConfig.make(T, Hd, E, K, 128, 0, 0.0, m.BF16)
    rng = np.random.default_rng(T)
    ids_np = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    ids_np[3, 1] = E                        # one id past the last expert
    ids = torch.from_numpy(ids_np).cuda()
    x = torch.randn(T, Hd, device="cuda").to(torch.bfloat16)
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(T * K, dtype=torch.int32, device="cuda")
    inv = torch.empty(T * K, dtype=torch.int32, device="cuda")
    x_perm = torch.empty(T * K, Hd, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(m.workspace_size(cfg), dtype=torch.uint8, device="cuda")
    assert dbg.moe_permute(ctypes.byref(cfg), _p(x), _p(ids), _p(counts), _p(offsets), _p(perm),
                           _p(inv), _p(x_perm), _p(ws), ctypes.c_size_t(ws.numel()), _s()) == 0
    assert dbg.moe_sync_check(_s()) == 6
    valid = ids_np[ids_np < E]
    np.testing.assert_array_equal(counts.cpu().numpy(), np.bincount(valid, minlength=E))
    assert int(inv.view(T, K)[3, 1]) == -1  # treated as not dispatched
    assert int(offsets[-1]) == len(valid)


def test_debug_build_reports_decreasing_group_offsets(dbg):
    import mixture_experts_layer_04_gb300 as m

    E, K, T, Hd, I = 4, 2, 64, 256, 128
    cfg = m.MoEConfig.make(T, Hd, E, K, I, 0, 0.0, m.BF16)
    x_perm = torch.randn(T * K, Hd, device="cuda").to(torch.bfloat16)
    w_gu = (torch.randn(E, 2 * I, Hd, device="cuda") * 0.02).to(torch.bfloat16)
    h = torch.full((T * K, I), 3.0, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(m.workspace_size(cfg), dtype=torch.uint8, device="cuda")
    bad = torch.tensor([0, 60, 40, 100, 128], dtype=torch.int32, device="cuda")
    assert dbg.moe_expert_gate_up(ctypes.byref(cfg), _p(x_perm), _p(bad), _p(w_gu), _p(h),
                                  _p(ws), ctypes.c_size_t(ws.numel()), _s()) == 0
    assert dbg.moe_sync_check(_s()) == 6
    assert bool((h == 3.0).all())           # the launch did nothing
    good = torch.tensor([0, 40, 60, 100, 128], dtype=torch.int32, device="cuda")
    assert dbg.moe_expert_gate_up(ctypes.byref(cfg), _p(x_perm), _p(good), _p(w_gu), _p(h),
                                  _p(ws), ctypes.c_size_t(ws.numel()), _s()) == 0
    assert dbg.moe_sync_check(_s()) == 0
    assert not bool((h == 3.0).all())
