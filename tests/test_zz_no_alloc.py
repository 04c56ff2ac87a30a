"""moe_permute_noalloc against moe_permute, through the C ABI.

moe_permute_noalloc serves callers that cannot allocate device memory (a server whose
device pools are all sized at start-up, a plug-in host that hands over only inputs and
outputs): it takes its scratch from a fixed array inside the library instead of a
caller workspace.  Two calls in a row, on different inputs, must each give exactly what
moe_permute gives with a workspace -- the second call also shows that what the first
call left in the shared array does not leak into the next result.  The file is named
to be collected last.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import mixture_experts_layer_04_gb300 as m
    from mixture_experts_layer_04_gb300 import build

    build.build()
    return m.load()


def _buffers(T, E, K, H, dtype):
    def i32(n):
        return torch.full((n,), -7, dtype=torch.int32, device="cuda")
    return dict(counts=i32(E), offsets=i32(E + 1), perm=i32(T * K), inv=i32(T * K),
                x_perm=torch.zeros(T * K, H, dtype=dtype, device="cuda"))


def _call(lib, name, cfg, x, ids, b, ws=None):
    p = ctypes.c_void_p
    args = [ctypes.byref(cfg), p(x.data_ptr()), p(ids.data_ptr()), p(b["counts"].data_ptr()),
            p(b["offsets"].data_ptr()), p(b["perm"].data_ptr()), p(b["inv"].data_ptr()),
            p(b["x_perm"].data_ptr())]
    if ws is not None:
        args += [p(ws.data_ptr()), ctypes.c_size_t(ws.numel())]
    args.append(p(torch.cuda.current_stream().cuda_stream))
    return getattr(lib, name)(*args)


@pytest.mark.parametrize("T,E,K,H,theta,dtype", [
    (4100, 256, 8, 128, 0.05, torch.bfloat16),
    (1000, 64, 4, 64, 0.0, torch.float32),
    # at most 256 tokens: the one-launch permutation, which needs no scratch words
    (200, 64, 4, 128, 0.0, torch.bfloat16),
])
def test_noalloc_matches_workspace_permute_twice(lib, T, E, K, H, theta, dtype):
    import mixture_experts_layer_04_gb300 as m

    cfg = m.MoEConfig.make(T, H, E, K, 64, 0, theta, m.BF16 if dtype == torch.bfloat16 else m.F32)
    ws = torch.empty(m.workspace_size(cfg), dtype=torch.uint8, device="cuda")
    for call in range(2):
        L = synth.random_logits(T, E, seed=100 + call)
        ids_np, _ = oracle.route(L.numpy(), K, theta)
        ids = torch.from_numpy(ids_np).cuda()
        x = torch.randn(T, H, generator=torch.Generator().manual_seed(call)).to(dtype).cuda()
        want = _buffers(T, E, K, H, dtype)
        got = _buffers(T, E, K, H, dtype)
        assert _call(lib, "moe_permute", cfg, x, ids, want, ws) == 0
        assert _call(lib, "moe_permute_noalloc", cfg, x, ids, got) == 0
        torch.cuda.synchronize()
        for k in want:
            assert torch.equal(got[k], want[k]), f"call {call}: {k} differs"
        assert int(got["offsets"][-1]) == int((ids_np >= 0).sum())


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    import mixture_experts_layer_04_gb300 as m

    max_words = 262144          # MOE_PERMUTE_NOALLOC_MAX_WORDS
    E = 1024
    T = (max_words // E + 1) * 256   # one 256-token block more than the array holds
    cfg = m.MoEConfig.make(T, 64, E, 2, 64, 0, 0.0, m.BF16)
    p = ctypes.c_void_p(256)         # never dereferenced: the call is rejected first
    st = lib.moe_permute_noalloc(ctypes.byref(cfg), p, p, p, p, p, p, p, None)
    assert st == 3                   # MOE_ERR_WORKSPACE
    ok = m.MoEConfig.make(T - 256, 64, E, 2, 64, 0, 0.0, m.BF16)
    assert np.ceil((T - 256) / 256) * E <= max_words
    st_small = lib.moe_permute_noalloc(ctypes.byref(ok), None, p, p, p, p, p, p, None)
    assert st_small == 1             # within the limit: reaches the pointer checks instead
