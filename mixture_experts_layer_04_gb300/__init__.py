"""Thin Python binding of libmoe_gb300 (the C ABI declared in include/moe.h).

Argument marshalling only: every step of the MoE layer runs in the library's CUDA
kernels.  PyTorch supplies device memory (tensors), streams and the current device.
Functions take torch CUDA tensors (or raw device addresses as ints, or None for NULL)
and raise ``MoEError`` when the library returns a status other than MOE_OK.

There is no fallback: if the shared library has not been built, or cannot be
loaded, every call raises.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

__all__ = [
    "MoEConfig", "MoEError", "F32", "BF16", "FLAG_FUSED_COMBINE", "FLAG_CAPACITY", "FLAG_FP8", "library_path", "load", "workspace_size",
    "route", "permute", "permute_noalloc", "grouped_ffn", "expert_gate_up", "expert_gate_up_gather", "quantize_fp8", "expert_gate_up_fp8", "expert_down_fp8", "layer_forward_fp8", "expert_down", "combine", "layer_forward", "workspace_views",
    "sync_check", "debug_wait_timeout", "status_string", "version",
]

F32 = 0
BF16 = 1
# moe_config_t.flags: fuse the combine into the down projection (bf16 layers; y is then
# correct to fp32 rounding but not bitwise reproducible run to run)
FLAG_FUSED_COMBINE = 1
FLAG_CAPACITY = 2
FLAG_FP8 = 4

_STATUS = {
    0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
    4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT", 6: "MOE_ERR_INTERNAL", 7: "MOE_ERR_MISALIGNED",
}


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {_STATUS.get(status, status)}")


class MoEConfig(ctypes.Structure):
    """moe_config_t: T, H, E, K, I, I_shared, gate_threshold, dtype, flags."""

    _fields_ = [
        ("T", ctypes.c_int32), ("H", ctypes.c_int32), ("E", ctypes.c_int32),
        ("K", ctypes.c_int32), ("I", ctypes.c_int32), ("I_shared", ctypes.c_int32),
        ("gate_threshold", ctypes.c_float), ("dtype", ctypes.c_int32), ("flags", ctypes.c_uint32),
    ]

    @classmethod
    def make(cls, T, H, E, K, I, I_shared=0, gate_threshold=0.0, dtype=BF16, flags=0):
        return cls(T, H, E, K, I, I_shared, gate_threshold, dtype, flags)

    def __repr__(self):
        return (f"MoEConfig(T={self.T}, H={self.H}, E={self.E}, K={self.K}, I={self.I}, "
                f"I_shared={self.I_shared}, theta={self.gate_threshold}, dtype={self.dtype})")


def library_path(debug: bool = False) -> str:
    """The release library, or with ``debug`` the bounds-checking build (-DMOE_DEBUG)."""
    return os.path.join(os.path.dirname(os.path.abspath(__file__)),
                        "_build_debug" if debug else "_build", "libmoe_gb300.so")


_LIB: Optional[ctypes.CDLL] = None

_P = ctypes.c_void_p
_CFG = ctypes.POINTER(MoEConfig)
_SIGS = {
    "moe_workspace_size": [_CFG, ctypes.POINTER(ctypes.c_size_t)],
    "moe_route": [_CFG, _P, _P, _P, _P, _P, _P, _P],
    "moe_permute": [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
    "moe_permute_noalloc": [_CFG, _P, _P, _P, _P, _P, _P, _P, _P],
    "moe_grouped_ffn": [_CFG, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
    "moe_expert_gate_up": [_CFG, _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
    "moe_expert_gate_up_gather": [_CFG, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
    "moe_quantize_fp8": [_P, ctypes.c_int64, ctypes.c_int32, _P, _P, _P],
    "moe_expert_gate_up_fp8": [_CFG, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
    "moe_expert_down_fp8": [_CFG, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
    "moe_layer_forward_fp8": [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                              ctypes.c_size_t, _P],
    "moe_expert_down": [_CFG, _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
    "moe_combine": [_CFG, _P, _P, _P, _P, _P, _P, _P],
    "moe_layer_forward": [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
    "moe_workspace_views": [_CFG, _P] + [ctypes.POINTER(_P)] * 10,
    "moe_sync_check": [_P],
    "moe_debug_wait_timeout": [ctypes.c_uint, _P, _P],
    "moe_status_string": [ctypes.c_int],
    "moe_version": [],
    "moe_kernel_launch_count": [],
    "moe_debug_set_fault": [ctypes.c_char_p, ctypes.c_int],
}


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libmoe_gb300.so (built by ``build.py``); raises if it is missing."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = path or library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libmoe_gb300.so not built ({path}); run "
                           "`python -c 'import __graft_entry__ as g; g.build()'` first")
    _LIB = _open(path)
    return _LIB


def _open(path: str) -> ctypes.CDLL:
    lib = ctypes.CDLL(path)
    for name, args in _SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = (ctypes.c_char_p if name in ("moe_status_string", "moe_version") else
                      ctypes.c_ulonglong if name == "moe_kernel_launch_count" else ctypes.c_int)
    return lib


def load_debug() -> ctypes.CDLL:
    """A handle on the bounds-checking build (``build.build(debug=True)``), separate from
    the release library that ``load()`` returns; raises if it is not built."""
    path = library_path(debug=True)
    if not os.path.exists(path):
        raise RuntimeError(f"debug build of libmoe_gb300.so missing ({path})")
    return _open(path)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str):
    if status != 0:
        raise MoEError(status, where)


def status_string(status: int) -> str:
    return load().moe_status_string(status).decode()


def version() -> str:
    return load().moe_version().decode()


def kernel_launch_count() -> int:
    """Kernels the library has launched in this process (moe_kernel_launch_count)."""
    return int(load().moe_kernel_launch_count())


def debug_set_fault(point: Optional[str], n: int = 1) -> None:
    """Arm (or with point None, disarm) the host-side fault injector: the n-th pass through
    `point` returns MOE_ERR_CUDA (moe_debug_set_fault)."""
    _check(load().moe_debug_set_fault(point.encode() if point else None, int(n)),
           "moe_debug_set_fault")


def workspace_size(cfg: MoEConfig) -> int:
    n = ctypes.c_size_t(0)
    _check(load().moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)), "moe_workspace_size")
    return n.value


def route(cfg, x, w_router, router_bias, logits, topk_ids, topk_w, stream=None):
    _check(load().moe_route(ctypes.byref(cfg), _ptr(x), _ptr(w_router), _ptr(router_bias),
                            _ptr(logits), _ptr(topk_ids), _ptr(topk_w), _stream(stream)),
           "moe_route")


def permute(cfg, x, topk_ids, counts, offsets, perm, inv, x_perm, ws, ws_bytes=None, stream=None):
    nb = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check(load().moe_permute(ctypes.byref(cfg), _ptr(x), _ptr(topk_ids), _ptr(counts),
                              _ptr(offsets), _ptr(perm), _ptr(inv), _ptr(x_perm), _ptr(ws), nb,
                              _stream(stream)), "moe_permute")


def permute_noalloc(cfg, x, topk_ids, counts, offsets, perm, inv, x_perm, stream=None):
    """moe_permute for callers that cannot allocate: no workspace; the library's fixed
    scratch array is used instead (shared by all calls on a device, so overlapping calls
    must be serialised by the caller)."""
    _check(load().moe_permute_noalloc(ctypes.byref(cfg), _ptr(x), _ptr(topk_ids), _ptr(counts),
                                      _ptr(offsets), _ptr(perm), _ptr(inv), _ptr(x_perm),
                                      _stream(stream)), "moe_permute_noalloc")


def grouped_ffn(cfg, x_perm, offsets, w_gate_up, w_down, out_perm, ws, ws_bytes=None, stream=None):
    nb = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check(load().moe_grouped_ffn(ctypes.byref(cfg), _ptr(x_perm), _ptr(offsets), _ptr(w_gate_up),
                                  _ptr(w_down), _ptr(out_perm), _ptr(ws), nb, _stream(stream)),
           "moe_grouped_ffn")


def expert_gate_up(cfg, x_perm, offsets, w_gate_up, h, ws, ws_bytes=None, stream=None):
    nb = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check(load().moe_expert_gate_up(ctypes.byref(cfg), _ptr(x_perm), _ptr(offsets),
                                     _ptr(w_gate_up), _ptr(h), _ptr(ws), nb, _stream(stream)),
           "moe_expert_gate_up")


def expert_gate_up_gather(cfg, x, perm, offsets, w_gate_up, h, ws, ws_bytes=None, stream=None):
    nb = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check(load().moe_expert_gate_up_gather(ctypes.byref(cfg), _ptr(x), _ptr(perm), _ptr(offsets),
                                            _ptr(w_gate_up), _ptr(h), _ptr(ws), nb,
                                            _stream(stream)),
           "moe_expert_gate_up_gather")


def quantize_fp8(x, codes, scales, stream=None):
    """Per-row E4M3 codes and float32 scales of a bf16 [rows, cols] tensor."""
    rows, cols = x.shape[0], x.numel() // max(1, x.shape[0])
    _check(load().moe_quantize_fp8(_ptr(x), rows, cols, _ptr(codes), _ptr(scales), _stream(stream)),
           "moe_quantize_fp8")


def expert_gate_up_fp8(cfg, x_codes, x_scales, offsets, w_codes, w_scales, h, ws, ws_bytes=None,
                       stream=None):
    nb = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check(load().moe_expert_gate_up_fp8(ctypes.byref(cfg), _ptr(x_codes), _ptr(x_scales),
                                         _ptr(offsets), _ptr(w_codes), _ptr(w_scales), _ptr(h),
                                         _ptr(ws), nb, _stream(stream)),
           "moe_expert_gate_up_fp8")


def expert_down_fp8(cfg, h_codes, h_scales, offsets, w_codes, w_scales, out_perm, ws,
                    ws_bytes=None, stream=None):
    nb = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check(load().moe_expert_down_fp8(ctypes.byref(cfg), _ptr(h_codes), _ptr(h_scales),
                                      _ptr(offsets), _ptr(w_codes), _ptr(w_scales),
                                      _ptr(out_perm), _ptr(ws), nb, _stream(stream)),
           "moe_expert_down_fp8")


def layer_forward_fp8(cfg, x, w_router, router_bias, w_gate_up_codes, w_gate_up_scales,
                      w_down_codes, w_down_scales, w_shared_gate_up, w_shared_down, y, y_f32, ws,
                      ws_bytes=None, stream=None):
    nb = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check(load().moe_layer_forward_fp8(
        ctypes.byref(cfg), _ptr(x), _ptr(w_router), _ptr(router_bias), _ptr(w_gate_up_codes),
        _ptr(w_gate_up_scales), _ptr(w_down_codes), _ptr(w_down_scales), _ptr(w_shared_gate_up),
        _ptr(w_shared_down), _ptr(y), _ptr(y_f32), _ptr(ws), nb, _stream(stream)),
        "moe_layer_forward_fp8")


def expert_down(cfg, h, offsets, w_down, out_perm, ws, ws_bytes=None, stream=None):
    nb = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check(load().moe_expert_down(ctypes.byref(cfg), _ptr(h), _ptr(offsets), _ptr(w_down),
                                  _ptr(out_perm), _ptr(ws), nb, _stream(stream)),
           "moe_expert_down")


def combine(cfg, out_perm, inv, topk_w, shared_out, y, y_f32=None, stream=None):
    _check(load().moe_combine(ctypes.byref(cfg), _ptr(out_perm), _ptr(inv), _ptr(topk_w),
                              _ptr(shared_out), _ptr(y), _ptr(y_f32), _stream(stream)),
           "moe_combine")


def layer_forward(cfg, x, w_router, router_bias, w_gate_up, w_down, w_shared_gate_up,
                  w_shared_down, y, y_f32, ws, ws_bytes=None, stream=None):
    nb = ws.numel() * ws.element_size() if ws_bytes is None else ws_bytes
    _check(load().moe_layer_forward(ctypes.byref(cfg), _ptr(x), _ptr(w_router), _ptr(router_bias),
                                    _ptr(w_gate_up), _ptr(w_down), _ptr(w_shared_gate_up),
                                    _ptr(w_shared_down), _ptr(y), _ptr(y_f32), _ptr(ws), nb,
                                    _stream(stream)), "moe_layer_forward")


def workspace_views(cfg, ws) -> dict:
    """Device addresses (ints) of the intermediates a moe_layer_forward left in `ws`."""
    names = ["logits", "topk_ids", "topk_w", "counts", "offsets", "perm", "inv", "x_perm",
             "out_perm", "shared_out"]
    outs = [_P() for _ in names]
    _check(load().moe_workspace_views(ctypes.byref(cfg), _ptr(ws), *[ctypes.byref(o) for o in outs]),
           "moe_workspace_views")
    return {n: o.value for n, o in zip(names, outs)}


def debug_wait_timeout(limit_us, done, stream=None):
    """Self-test of the bounded device-side waits: a wait that nothing completes gives up
    after limit_us and records MOE_ERR_TIMEOUT for the next sync_check()."""
    _check(load().moe_debug_wait_timeout(limit_us, _ptr(done), _stream(stream)),
           "moe_debug_wait_timeout")


def sync_check(stream=None):
    _check(load().moe_sync_check(_stream(stream)), "moe_sync_check")
