"""The host-side fault injector and the bounds-checking build, without a GPU.

moe_debug_set_fault (or MOE_FAULT=<point>:<n> in the environment when the library loads)
makes the n-th pass through a named point return MOE_ERR_CUDA there, as a failed launch
would, and then disarms; a caller can rehearse its clean-up after a failed call.  Page
"MoE大模型的智能调度…" §3.2 recounts production failures of the routing step (trap 2: an
out-of-memory crash); these tests fail on the host only, no GPU is involved.  An entry
point's own fault is checked before anything else, so no output is written; the next call
runs normally.  The debug build (-DMOE_DEBUG) must compile and export the same C ABI.
"""

import ctypes
import os
import subprocess
import sys

import pytest

from tests.conftest import ROOT
from tests.test_abi_cpu import declared_functions

import mixture_experts_layer_04_gb300 as moe
from mixture_experts_layer_04_gb300 import build as moe_build

OK, INVALID, CUDA = 0, 1, 4


@pytest.fixture(scope="module")
def lib():
    moe_build.build()
    return moe.load()


@pytest.fixture(autouse=True)
def disarm(lib):
    lib.moe_debug_set_fault(None, 0)
    yield
    lib.moe_debug_set_fault(None, 0)


def _cfg(T=64):
    return moe.MoEConfig.make(T, 256, 8, 2, 128, 0, 0.0, moe.BF16)


def test_unknown_point_is_rejected(lib):
    assert lib.moe_debug_set_fault(b"moe_no_such_call", 1) == INVALID
    assert lib.moe_debug_set_fault(b"moe_layer_forward.nowhere", 1) == INVALID
    assert lib.moe_debug_set_fault(b"moe_route", 1) == OK
    assert lib.moe_debug_set_fault(None, 0) == OK


def test_nth_call_fails_once_and_leaves_its_output_untouched(lib):
    c = _cfg()
    size = ctypes.c_size_t(0)
    assert lib.moe_workspace_size(ctypes.byref(c), ctypes.byref(size)) == OK
    want = size.value
    assert lib.moe_debug_set_fault(b"moe_workspace_size", 2) == OK
    out = ctypes.c_size_t(12345)
    assert lib.moe_workspace_size(ctypes.byref(c), ctypes.byref(out)) == OK    # 1st: passes
    assert out.value == want
    out.value = 12345
    assert lib.moe_workspace_size(ctypes.byref(c), ctypes.byref(out)) == CUDA  # 2nd: injected
    assert out.value == 12345                                                 # untouched
    assert lib.moe_workspace_size(ctypes.byref(c), ctypes.byref(out)) == OK    # disarmed
    assert out.value == want


def test_fault_precedes_argument_checks_and_other_points_pass(lib):
    c = _cfg(T=0)   # an empty batch is a valid no-op, so these calls need no GPU
    A = ctypes.c_void_p(0x7000_0000_0000)
    args = (ctypes.byref(c), A, A, None, A, A, None, None, A, None, A, ctypes.c_size_t(1 << 30), None)
    assert lib.moe_debug_set_fault(b"moe_layer_forward", 1) == OK
    assert lib.moe_route(ctypes.byref(c), A, A, None, A, A, A, None) == OK    # another point
    assert lib.moe_layer_forward(*args) == CUDA
    assert lib.moe_layer_forward(*args) == OK
    # the binding raises the status as MoEError
    moe.debug_set_fault("moe_route", 1)
    with pytest.raises(moe.MoEError) as ei:
        moe.route(c, None, None, None, None, None, None, stream=0)
    assert ei.value.status == CUDA
    moe.route(c, None, None, None, None, None, None, stream=0)
    with pytest.raises(moe.MoEError):
        moe.debug_set_fault("not_a_point", 1)


_CHILD = """
import ctypes, sys
sys.path.insert(0, {root!r})
import mixture_experts_layer_04_gb300 as moe
lib = moe.load()
c = moe.MoEConfig.make(0, 256, 8, 2, 128, 0, 0.0, moe.BF16)
A = ctypes.c_void_p(0x7000_0000_0000)
print(lib.moe_route(ctypes.byref(c), A, A, None, A, A, A, None),
      lib.moe_route(ctypes.byref(c), A, A, None, A, A, A, None),
      lib.moe_route(ctypes.byref(c), A, A, None, A, A, A, None))
"""


@pytest.mark.parametrize("spec,want,warn", [
    ("moe_route:2", "0 4 0", False),
    ("moe_route", "0 0 0", True),           # no count: ignored, with a warning
    ("moe_nothing:1", "0 0 0", True),       # unknown point: ignored, with a warning
])
def test_environment_arms_the_fault_at_load(lib, spec, want, warn):
    env = dict(os.environ, MOE_FAULT=spec, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", _CHILD.format(root=ROOT)], env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.split("\n")[-2].strip() == want
    assert ("MOE_FAULT" in r.stderr) == warn


def test_debug_build_exports_the_same_abi():
    path = moe_build.build(debug=True)
    assert path == moe.library_path(debug=True) and os.path.exists(path)
    dbg = moe.load_debug()
    for name in declared_functions():
        assert hasattr(dbg, name), name
    assert "sm_103a" in dbg.moe_version().decode()
