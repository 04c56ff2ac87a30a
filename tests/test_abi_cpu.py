"""Host-side checks of the C ABI (no GPU needed).

The library must build, load and export every function include/moe.h declares; the
workspace planner and the argument checks run on the host and must answer before any
CUDA call; on a machine without a usable GPU a valid call must fail loudly
(MOE_ERR_CUDA or MOE_ERR_UNSUPPORTED), never compute on the CPU.
"""

import ctypes
import os
import re

import pytest
import torch

from tests.conftest import ROOT

import mixture_experts_layer_04_gb300 as moe
from mixture_experts_layer_04_gb300 import build as moe_build

HEADER = os.path.join(ROOT, "include", "moe.h")

OK, INVALID, UNSUPPORTED, WORKSPACE, CUDA, TIMEOUT, INTERNAL, MISALIGNED = range(8)


@pytest.fixture(scope="module")
def lib():
    moe_build.build()
    return moe.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_stage_calls():
    names = declared_functions()
    for n in ["moe_route", "moe_permute", "moe_grouped_ffn", "moe_combine", "moe_layer_forward",
              "moe_workspace_size", "moe_expert_gate_up", "moe_expert_down", "moe_sync_check",
              "moe_status_string"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    assert moe.status_string(0) == "MOE_OK"
    assert moe.status_string(3) == "MOE_ERR_WORKSPACE"
    assert "sm_103a" in moe.version()


def cfg(**kw):
    base = dict(T=64, H=256, E=8, K=2, I=128, I_shared=0, gate_threshold=0.0, dtype=moe.BF16)
    base.update(kw)
    return moe.MoEConfig.make(**base)


def ws_size(c):
    n = ctypes.c_size_t(0)
    st = moe.load().moe_workspace_size(ctypes.byref(c), ctypes.byref(n))
    return st, n.value


@pytest.mark.parametrize("bad", [
    dict(K=0), dict(K=9), dict(E=2000, K=2), dict(K=17, E=32), dict(H=100), dict(I=96),
    dict(I_shared=32), dict(T=-1), dict(gate_threshold=1.0), dict(gate_threshold=-0.1),
    dict(dtype=7), dict(flags=8), dict(flags=0x80000000),
])
def test_invalid_configs_are_rejected(lib, bad):
    st, _ = ws_size(cfg(**bad))
    assert st == INVALID


def test_workspace_size_grows_with_tokens(lib):
    sizes = [ws_size(cfg(T=t))[1] for t in (0, 1, 64, 1000)]
    assert all(ws_size(cfg(T=t))[0] == OK for t in (0, 1, 64, 1000))
    assert sizes == sorted(sizes) and sizes[-1] > sizes[0]
    # the routed intermediates of a Mixtral-shaped prefill are all in the workspace
    big = ws_size(cfg(T=4096, H=4096, E=8, K=2, I=14336))[1]
    assert big >= 4096 * 2 * (4096 * 2 + 14336 * 2 + 4096 * 4)


def _p(v):
    return ctypes.c_void_p(v)


def test_argument_errors_are_host_side(lib):
    c = cfg()
    A = 0x7000_0000_0000  # never dereferenced: every call below fails validation first
    # null outputs
    assert lib.moe_route(ctypes.byref(c), _p(A), _p(A), None, None, _p(A), _p(A), None) == INVALID
    # misaligned pointer
    assert lib.moe_route(ctypes.byref(c), _p(A + 4), _p(A), None, _p(A), _p(A), _p(A), None) == MISALIGNED
    # workspace too small / missing
    need = ws_size(c)[1]
    assert lib.moe_permute(ctypes.byref(c), _p(A), _p(A), _p(A), _p(A), _p(A), _p(A), _p(A),
                           _p(A), need - 1, None) == WORKSPACE
    assert lib.moe_layer_forward(ctypes.byref(c), _p(A), _p(A), None, _p(A), _p(A), None, None,
                                 _p(A), None, None, need, None) == WORKSPACE
    # shared-expert pointers must match I_shared
    cs = cfg(I_shared=128)
    assert lib.moe_layer_forward(ctypes.byref(cs), _p(A), _p(A), None, _p(A), _p(A), None, None,
                                 _p(A), None, _p(A), ws_size(cs)[1], None) == INVALID
    assert lib.moe_grouped_ffn(ctypes.byref(c), None, _p(A), _p(A), _p(A), _p(A), _p(A), need,
                               None) == INVALID
    assert lib.moe_combine(ctypes.byref(c), _p(A), _p(A), _p(A), None, _p(A + 8), None, None) == MISALIGNED


def test_row_gather_gate_up_is_bf16_only(lib):
    c = cfg(dtype=moe.F32)
    A = 0x7000_0000_0000
    need = ws_size(c)[1]
    assert lib.moe_expert_gate_up_gather(ctypes.byref(c), _p(A), _p(A), _p(A), _p(A), _p(A), _p(A),
                                         need, None) == UNSUPPORTED
    cb = cfg()
    assert lib.moe_expert_gate_up_gather(ctypes.byref(cb), _p(A), None, _p(A), _p(A), _p(A), _p(A),
                                         ws_size(cb)[1], None) == INVALID


def test_zero_tokens_is_a_noop_without_gpu(lib):
    c = cfg(T=0)
    A = 0x7000_0000_0000
    need = ws_size(c)[1]
    assert lib.moe_layer_forward(ctypes.byref(c), _p(A), _p(A), None, _p(A), _p(A), None, None,
                                 _p(A), None, _p(A), need, None) == OK
    assert lib.moe_route(ctypes.byref(c), _p(A), _p(A), None, _p(A), _p(A), _p(A), None) == OK


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks behaviour without a GPU")
def test_valid_call_without_gpu_fails_loudly(lib):
    c = cfg()
    A = 0x7000_0000_0000
    st = lib.moe_route(ctypes.byref(c), _p(A), _p(A), None, _p(A), _p(A), _p(A), None)
    assert st in (CUDA, UNSUPPORTED)
