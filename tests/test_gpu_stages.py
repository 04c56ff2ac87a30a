"""GPU parity of every stage of the MoE layer against the CPU oracle, through the C ABI.

Each stage is fed the same inputs as the oracle stage (seeded, synthetic), at sizes the
oracle finishes in seconds that still span several tiles and a ragged tail:
  * routing from given float32 logits: ids bit-exact (ties to the lower expert), gates
    to 1e-5; tokens whose gate lies within rounding of the drop threshold are only
    checked for validity;
  * router logits (tensor-core and SIMT paths): within fp32 accumulation error, ids
    bit-exact on tokens without a near-tie;
  * permutation: counts, offsets, perm, inv bit-exact, x_perm rows bitwise copies, rows
    past the kept count untouched;
  * gate/up + SwiGLU, down projection, and both: within the stated tolerances, rows
    of neighbouring experts and padding never leak into a group's output;
  * combine: fp32 sum within 1e-5, the bf16 output is the RNE rounding of it.
"""

import numpy as np
import pytest
import torch

import oracle
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


def _cfg(moe, T, H_, E, K, I=64, Is=0, theta=0.0, dtype="bf16"):
    return moe.MoEConfig.make(T, H_, E, K, I, Is, theta, moe.BF16 if dtype == "bf16" else moe.F32)


def _logits(T, E, seed, ties):
    L = synth.random_logits(T, E, seed=seed, scale=1.5)
    if ties:
        L[::3] = torch.round(L[::3] * 2) / 2     # exact ties in every third token
        L[1::7] = 0.25                           # all-equal tokens
    return L


ROUTE_CASES = [
    (1, 4, 1, 0.0), (37, 8, 2, 0.0), (300, 128, 8, 0.0), (1000, 256, 8, 0.05),
    (513, 1024, 16, 0.02), (64, 16, 16, 0.0), (200, 64, 4, 0.2), (129, 33, 3, 0.1),
]


@pytest.mark.parametrize("T,E,K,theta", ROUTE_CASES)
@pytest.mark.parametrize("ties", [False, True])
def test_route_from_logits_bit_exact(moe, T, E, K, theta, ties):
    L = _logits(T, E, seed=T + E, ties=ties)
    c = _cfg(moe, T, 64, E, K, theta=theta)
    Lg = L.cuda()
    ids = torch.full((T, K), -9, dtype=torch.int32, device="cuda")
    w = torch.full((T, K), -9.0, dtype=torch.float32, device="cuda")
    moe.route(c, None, None, None, Lg, ids, w)
    torch.cuda.synchronize()
    ids_ref, w_ref = oracle.route(L.numpy(), K, theta)
    amb = H.compare_routing(L.numpy(), ids.cpu().numpy(), w.cpu().numpy(), ids_ref, w_ref, K,
                            theta, margin=None)
    assert amb.mean() < 0.01
    assert torch.equal(Lg.cpu(), L)              # logits are an input here: untouched


def _skewed_logits(T, E, skew, seed):
    L = synth.random_logits(T, E, seed=seed)
    if skew == "normal":
        L = L + torch.randn(E, generator=torch.Generator().manual_seed(seed)) * 1.0
    elif skew == "zipf":
        r = torch.randperm(E, generator=torch.Generator().manual_seed(seed)).double() + 1
        L = L + (-1.1 * torch.log(r)).float()
    elif skew == "one":
        L[:, E // 2] += 50.0
    return L


CAPACITY_CASES = [
    # T, E, K, theta, skew
    (1, 8, 2, 0.0, "none"), (37, 16, 4, 0.0, "one"), (300, 8, 2, 0.1, "zipf"),
    (1000, 64, 8, 0.0, "normal"), (5000, 128, 8, 0.0, "zipf"), (2048, 256, 8, 0.05, "zipf"),
    (600, 1024, 16, 0.0, "normal"), (700, 4, 2, 0.0, "one"),
]


@pytest.mark.parametrize("T,E,K,theta,skew", CAPACITY_CASES)
def test_capacity_route_equals_oracle(moe, T, E, K, theta, skew):
    L = _skewed_logits(T, E, skew, seed=T + 3 * E)
    c = moe.MoEConfig.make(T, 64, E, K, 64, 0, theta, moe.BF16, moe.FLAG_CAPACITY)
    Lg = L.cuda()
    ids = torch.full((T, K), -9, dtype=torch.int32, device="cuda")
    w = torch.full((T, K), -9.0, dtype=torch.float32, device="cuda")
    moe.route(c, None, None, None, Lg, ids, w)
    torch.cuda.synchronize()
    moe.sync_check()
    ids_ref, w_ref = oracle.route_capacity(L.numpy(), K, theta)
    # the gate drop is an fp32 decision on the GPU and fp64 in the oracle: these inputs
    # keep every gate clear of the threshold, so both take the same decisions
    assert H.capacity_gate_margin(L.numpy(), K, theta, ids_ref) > 1e-5
    np.testing.assert_array_equal(ids.cpu().numpy(), ids_ref)
    np.testing.assert_allclose(w.cpu().numpy(), w_ref, rtol=0, atol=1e-5)
    counts = np.bincount(ids_ref[ids_ref >= 0], minlength=E)
    assert counts.max() <= oracle.capacity(T, K, E)
    if skew != "none":  # the capacity binds: the result differs from plain routing
        assert not np.array_equal(ids_ref, oracle.route(L.numpy(), K, theta)[0])


ROUTER_CASES = [
    # T, H, E, dtype, bias   (bf16 with T >= 256 and E % 16 == 0 uses the tensor cores)
    (1024, 512, 128, "bf16", "normal"),
    (257, 256, 256, "bf16", "zipf"),
    (300, 1024, 8, "bf16", "none"),
    (64, 2048, 128, "bf16", "normal"),
    (16, 7168, 256, "bf16", "zipf"),           # one slice of 896 units: several bursts
    (100, 1088, 24, "bf16", "normal"),
    (256, 512, 8, "f32", "none"),
    (3, 192, 40, "f32", "normal"),
]


@pytest.mark.parametrize("T,H_,E,dtype,bias", ROUTER_CASES)
def test_router_logits_and_selection(moe, T, H_, E, dtype, bias):
    K = min(8, E)
    shape = synth.MoEShape("r", T=T, H=H_, E=E, K=K, I=64, dtype=dtype, bias=bias, seed=11)
    inp = synth.make_inputs(shape, device="cuda", weights=False)
    c = _cfg(moe, T, H_, E, K, dtype=dtype)
    logits = torch.empty(T, E, dtype=torch.float32, device="cuda")
    ids = torch.empty(T, K, dtype=torch.int32, device="cuda")
    w = torch.empty(T, K, dtype=torch.float32, device="cuda")
    moe.route(c, inp["x"], inp["w_router"], inp["router_bias"], logits, ids, w)
    torch.cuda.synchronize()
    b = inp["router_bias"].cpu().numpy() if inp["router_bias"] is not None else None
    L_ref = oracle.router_logits(H.f64(inp["x"]), H.f64(inp["w_router"]), b)
    got = logits.double().cpu().numpy()
    assert np.abs(got - L_ref).max() <= 1e-4 * max(1.0, np.abs(L_ref).max())
    L32 = L_ref.astype(np.float32)
    ids_ref, w_ref = oracle.route(L32, K, 0.0)
    amb = H.compare_routing(L32, ids.cpu().numpy(), w.cpu().numpy(), ids_ref, w_ref, K, 0.0)
    assert amb.mean() < 0.02


@pytest.mark.parametrize("T,H_,E,K,theta,dup", [
    (512, 256, 128, 8, 0.0, False),
    (300, 512, 256, 16, 0.05, True),    # K = 16, gate drop, duplicated experts (exact ties)
    (256, 128, 48, 6, 0.1, True),       # E = 48: the 64-column tile masks 16 columns
    (1000, 256, 32, 1, 0.0, False),
    (384, 128, 64, 4, 0.2, True),
    (260, 64, 96, 8, 0.0, "all"),       # every expert has the same weights: all logits tie
])
def test_tensor_core_router_topk_equals_warp_topk(moe, T, H_, E, K, theta, dup):
    """The tensor-core router takes the top-k in its epilogue, one thread per token; given
    the logits it wrote, the ids and gates equal the warp top-k's (moe_route from logits)
    bit for bit, ties going to the lower expert id."""
    shape = synth.MoEShape("r", T=T, H=H_, E=E, K=K, I=64, dtype="bf16", bias="normal", seed=5)
    inp = synth.make_inputs(shape, device="cuda", weights=False)
    wr = inp["w_router"].clone()
    bias = inp["router_bias"]
    if dup == "all":
        wr[:] = wr[0]
        bias = None
    elif dup:
        wr[1::3] = wr[0::3][: wr[1::3].shape[0]]   # expert 3j+1 copies expert 3j
        bias = None
    c = _cfg(moe, T, H_, E, K, theta=theta)
    logits = torch.empty(T, E, dtype=torch.float32, device="cuda")
    ids = torch.full((T, K), -9, dtype=torch.int32, device="cuda")
    w = torch.full((T, K), -9.0, dtype=torch.float32, device="cuda")
    moe.route(c, inp["x"], wr, bias, logits, ids, w)
    ids2 = torch.full((T, K), -9, dtype=torch.int32, device="cuda")
    w2 = torch.full((T, K), -9.0, dtype=torch.float32, device="cuda")
    moe.route(c, None, None, None, logits, ids2, w2)
    torch.cuda.synchronize()
    assert torch.equal(ids, ids2)
    assert torch.equal(w, w2)
    if dup == "all":
        assert (ids.cpu() == torch.arange(K, dtype=torch.int32)).all()
    b = bias.cpu().numpy() if bias is not None else None
    L_ref = oracle.router_logits(H.f64(inp["x"]), H.f64(wr), b)
    assert np.abs(logits.double().cpu().numpy() - L_ref).max() <= 1e-4 * max(1.0, np.abs(L_ref).max())


PERMUTE_CASES = [
    # T, E, K, theta, H, skew
    (1, 4, 2, 0.0, 64, "none"), (255, 8, 2, 0.0, 128, "none"), (257, 8, 2, 0.0, 128, "none"),
    (1000, 128, 8, 0.05, 64, "normal"), (4100, 256, 8, 0.05, 64, "zipf"),
    (700, 1024, 16, 0.02, 64, "normal"), (300, 16, 16, 0.0, 64, "none"),
    (513, 32, 1, 0.0, 64, "one"), (999, 64, 4, 0.1, 64, "empties"),
]


def _skewed_ids(T, E, K, theta, skew, seed):
    L = synth.random_logits(T, E, seed=seed)
    if skew == "normal":
        L = L + torch.randn(E, generator=torch.Generator().manual_seed(seed)) * 1.0
    elif skew == "zipf":
        r = torch.randperm(E, generator=torch.Generator().manual_seed(seed)).double() + 1
        L = L + (-1.1 * torch.log(r)).float()
    elif skew == "one":
        L[:, E // 2] += 50.0
    elif skew == "empties":
        L[:, ::3] -= 1e4
    return oracle.route(L.numpy(), K, theta)


@pytest.mark.parametrize("T,E,K,theta,H_,skew", PERMUTE_CASES)
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_permute_bit_exact(moe, T, E, K, theta, H_, skew, dtype):
    ids_ref, _ = _skewed_ids(T, E, K, theta, skew, seed=T * 7 + E)
    counts_r, offsets_r, perm_r, inv_r = oracle.permute(ids_ref, E)
    M = int(offsets_r[-1])
    c = _cfg(moe, T, H_, E, K, theta=theta, dtype=dtype)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    x = torch.randn(T, H_, generator=torch.Generator().manual_seed(5)).to(tdt).cuda()
    ids = torch.from_numpy(ids_ref).cuda()
    counts = torch.full((E,), -7, dtype=torch.int32, device="cuda")
    offsets = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    perm = torch.full((T * K,), -7, dtype=torch.int32, device="cuda")
    inv = torch.full((T * K,), -7, dtype=torch.int32, device="cuda")
    x_perm = torch.full((T * K, H_), 3.0, dtype=tdt, device="cuda")
    ws = torch.empty(moe.workspace_size(c), dtype=torch.uint8, device="cuda")
    moe.permute(c, x, ids, counts, offsets, perm, inv, x_perm, ws)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(counts.cpu().numpy(), counts_r)
    np.testing.assert_array_equal(offsets.cpu().numpy(), offsets_r)
    np.testing.assert_array_equal(perm[:M].cpu().numpy(), perm_r)
    assert (perm[M:] == -7).all()
    np.testing.assert_array_equal(inv.view(T, K).cpu().numpy(), inv_r)
    assert torch.equal(x_perm[:M].cpu(), x.cpu()[torch.from_numpy(perm_r).long()])
    assert (x_perm[M:] == 3.0).all()


FFN_CASES = [
    # T, H, E, K, I, dtype, skew
    (300, 256, 8, 2, 128, "bf16", "none"),
    (1000, 512, 64, 4, 192, "bf16", "normal"),
    (129, 320, 16, 8, 256, "bf16", "empties"),
    (700, 256, 4, 1, 128, "bf16", "one"),
    (64, 256, 16, 8, 128, "bf16", "normal"),     # decode sizes: weights on the MMA's M side
    (8, 512, 128, 8, 192, "bf16", "none"),
    (128, 256, 8, 2, 256, "bf16", "one"),         # one expert gets 128 rows: two token tiles
    (1, 128, 4, 2, 64, "bf16", "none"),
    (33, 320, 8, 4, 128, "bf16", "empties"),
    (256, 512, 8, 2, 1024, "f32", "none"),
    (77, 128, 4, 3, 64, "f32", "normal"),
]


def _ffn_inputs(T, H_, E, K, I, dtype, skew, seed=1):
    ids, _ = _skewed_ids(T, E, K, 0.0, skew, seed=seed + T)
    counts, offsets, perm, inv = oracle.permute(ids, E)
    shape = synth.MoEShape("f", T=T, H=H_, E=E, K=K, I=I, dtype=dtype, seed=seed)
    inp = synth.make_inputs(shape, device="cuda")
    tdt = shape.torch_dtype
    M = int(offsets[-1])
    x_perm = torch.full((T * K, H_), float("nan"), dtype=tdt, device="cuda")  # padding = NaN
    x_perm[:M] = inp["x"][torch.from_numpy(perm).long().cuda()]
    return shape, inp, offsets, x_perm, M


@pytest.mark.parametrize("T,H_,E,K,I,dtype,skew", FFN_CASES)
def test_grouped_ffn_stages(moe, T, H_, E, K, I, dtype, skew):
    shape, inp, offsets, x_perm, M = _ffn_inputs(T, H_, E, K, I, dtype, skew)
    c = _cfg(moe, T, H_, E, K, I=I, dtype=dtype)
    tdt = shape.torch_dtype
    off = torch.from_numpy(offsets).cuda()
    ws = torch.empty(moe.workspace_size(c), dtype=torch.uint8, device="cuda")
    h = torch.full((T * K, I), -5.0, dtype=tdt, device="cuda")
    moe.expert_gate_up(c, x_perm, off, inp["w_gate_up"], h, ws)
    out = torch.full((T * K, H_), -5.0, dtype=torch.float32, device="cuda")
    moe.expert_down(c, h, off, inp["w_down"], out, ws)
    out2 = torch.full((T * K, H_), -5.0, dtype=torch.float32, device="cuda")
    moe.grouped_ffn(c, x_perm, off, inp["w_gate_up"], inp["w_down"], out2, ws)
    torch.cuda.synchronize()
    assert (h[M:] == -5.0).all() and (out[M:] == -5.0).all() and (out2[M:] == -5.0).all()
    xp = H.f64(x_perm[:M])
    h_gpu = H.f64(h[:M])
    o_gpu = out[:M].double().cpu().numpy()
    h_ref = np.zeros((M, I))
    o_of_hgpu = np.zeros((M, H_))
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 > r0:
            h_ref[r0:r1] = oracle.expert_gate_up(xp[r0:r1], H.f64(inp["w_gate_up"][e]))
            o_of_hgpu[r0:r1] = oracle.expert_down(h_gpu[r0:r1], H.f64(inp["w_down"][e]))
    if dtype == "bf16":
        # h is rounded once to bf16: half an ulp (2^-9 relative) plus fp32 accumulation
        assert (np.abs(h_gpu - h_ref) <= 2.0 ** -8 * np.abs(h_ref) + 1e-4).all()
        H.assert_close_y(o_gpu, o_of_hgpu, max_abs=1e-3, rel_l2=1e-5, what="down")
    else:
        H.assert_close_y(h_gpu, h_ref, max_abs=1e-4, rel_l2=1e-5, what="gate_up")
        H.assert_close_y(o_gpu, o_of_hgpu, max_abs=1e-4, rel_l2=1e-5, what="down")
    # the fused call equals the two stages, and the whole FFN matches the oracle
    assert torch.equal(out2[:M], out[:M])
    o_ref = oracle.grouped_ffn(xp, offsets, H.ExpertSlices(inp["w_gate_up"]),
                               H.ExpertSlices(inp["w_down"]))
    if dtype == "bf16":
        H.assert_close_y(o_gpu, o_ref[:M], what="grouped_ffn")
    else:
        H.assert_close_y(o_gpu, o_ref[:M], max_abs=H.Y32_MAX_ABS, rel_l2=H.Y32_REL_L2,
                         what="grouped_ffn")


# Groups of >= 768 rows on average run on CTA pairs (256-row tiles).  A group's last tile
# with r < 256 rows runs in swapped order when r rounds up to at most 192 token columns,
# else padded; these sizes give tails of 1, 33, 31, 192, 255 (padded), 0, 96 and 160 rows
# and one empty group.
PAIR_GROUPS = [769, 801, 1055, 1216, 0, 1279, 1024, 864, 928]


@pytest.mark.parametrize("H_,I", [(256, 128), (512, 320)])
def test_pair_tiles_with_swapped_tails(moe, H_, I):
    sizes = np.array(PAIR_GROUPS)
    E, K = len(sizes), 2
    M = int(sizes.sum())
    T = (M + 255) // K  # a few spare rows after the last group
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    shape = synth.MoEShape("pair", T=T, H=H_, E=E, K=K, I=I, seed=12)
    inp = synth.make_inputs(shape, device="cuda")
    gen = torch.Generator().manual_seed(13)
    x_perm = torch.full((T * K, H_), float("nan"), dtype=torch.bfloat16, device="cuda")
    x_perm[:M] = torch.randn(M, H_, generator=gen).to(torch.bfloat16).cuda()
    c = _cfg(moe, T, H_, E, K, I=I, dtype="bf16")
    off = torch.from_numpy(offsets).cuda()
    ws = torch.empty(moe.workspace_size(c), dtype=torch.uint8, device="cuda")
    h = torch.full((T * K, I), -5.0, dtype=torch.bfloat16, device="cuda")
    moe.expert_gate_up(c, x_perm, off, inp["w_gate_up"], h, ws)
    out = torch.full((T * K, H_), -5.0, dtype=torch.float32, device="cuda")
    moe.expert_down(c, h, off, inp["w_down"], out, ws)
    torch.cuda.synchronize()
    moe.sync_check()
    assert (h[M:] == -5.0).all() and (out[M:] == -5.0).all()
    xp = H.f64(x_perm[:M])
    h_gpu = H.f64(h[:M])
    h_ref = np.zeros((M, I))
    o_of_hgpu = np.zeros((M, H_))
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 > r0:
            h_ref[r0:r1] = oracle.expert_gate_up(xp[r0:r1], H.f64(inp["w_gate_up"][e]))
            o_of_hgpu[r0:r1] = oracle.expert_down(h_gpu[r0:r1], H.f64(inp["w_down"][e]))
    assert np.isfinite(h_gpu).all()
    assert (np.abs(h_gpu - h_ref) <= 2.0 ** -8 * np.abs(h_ref) + 1e-4).all()
    H.assert_close_y(out[:M].double().cpu().numpy(), o_of_hgpu, max_abs=1e-3, rel_l2=1e-5,
                     what="down")


def _e4m3_bytes(values):
    """The E4M3 bit patterns of float64 values that are exact E4M3 numbers."""
    return torch.from_numpy(np.asarray(values, dtype=np.float32)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()


# row lengths that take each of the quantiser's paths: rows held in registers (up to 4 or
# 8 16-byte units per lane, or 17-28 as at H = 7168) and rows read twice (4096, 14336)
@pytest.mark.parametrize("cols", [384, 2048, 4096, 7168, 14336, 72])
def test_quantize_fp8_bit_exact(moe, cols):
    gen = torch.Generator().manual_seed(31)
    rows = 300 if cols <= 4096 else 64
    a = torch.randn(rows, cols, generator=gen) * torch.rand(rows, 1, generator=gen) * 20
    a[7] = 0.0                      # an all-zero row: scale 1
    a[11, 5] = 1e4                  # one large value: the rest of the row goes subnormal
    a[13] = 1e-6 * torch.randn(cols, generator=gen)
    x = a.to(torch.bfloat16).cuda()
    codes = torch.full((rows, cols), 0x55, dtype=torch.uint8, device="cuda")
    scales = torch.full((rows,), -1.0, dtype=torch.float32, device="cuda")
    moe.quantize_fp8(x, codes, scales)
    torch.cuda.synchronize()
    ref_codes, ref_scales = oracle.quantize_rows_fp8(x.float().cpu().numpy())
    np.testing.assert_array_equal(scales.cpu().numpy(), ref_scales)
    np.testing.assert_array_equal(codes.cpu().numpy(), _e4m3_bytes(ref_codes))


FP8_CASES = [
    # T, H, E, K, I, skew   (T <= 128: the decode-sized, swapped tiles)
    (300, 256, 8, 2, 128, "none"), (1000, 512, 64, 4, 192, "normal"), (129, 384, 16, 8, 320, "empties"),
    (64, 256, 16, 8, 128, "normal"), (8, 512, 32, 4, 128, "none"), (1, 256, 8, 2, 64, "none"),
]


@pytest.mark.parametrize("T,H_,E,K,I,skew", FP8_CASES)
def test_gate_up_fp8_equals_oracle(moe, T, H_, E, K, I, skew):
    """E4M3 activations and weights with per-row scales, quantised on the GPU (bit-exact
    against the oracle's quantiser), then the FP8 gate/up against the oracle's FP8 gate/up
    on the same codes: fp32 accumulation of exact products, h rounded once to bf16."""
    shape, inp, offsets, x_perm, M = _ffn_inputs(T, H_, E, K, I, "bf16", skew)
    x_perm[M:] = 0
    c = _cfg(moe, T, H_, E, K, I=I, dtype="bf16")
    ws = torch.empty(moe.workspace_size(c), dtype=torch.uint8, device="cuda")
    xq = torch.empty(T * K, H_, dtype=torch.uint8, device="cuda")
    xs = torch.empty(T * K, dtype=torch.float32, device="cuda")
    moe.quantize_fp8(x_perm, xq, xs)
    wq = torch.empty(E, 2 * I, H_, dtype=torch.uint8, device="cuda")
    wsc = torch.empty(E, 2 * I, dtype=torch.float32, device="cuda")
    moe.quantize_fp8(inp["w_gate_up"].reshape(E * 2 * I, H_), wq, wsc)
    h = torch.full((T * K, I), -5.0, dtype=torch.bfloat16, device="cuda")
    moe.expert_gate_up_fp8(c, xq, xs, torch.from_numpy(offsets).cuda(), wq, wsc, h, ws)
    torch.cuda.synchronize()
    moe.sync_check()
    assert (h[M:] == -5.0).all()
    xc, xsc = oracle.quantize_rows_fp8(x_perm[:M].float().cpu().numpy())
    np.testing.assert_array_equal(xq[:M].cpu().numpy(), _e4m3_bytes(xc))
    np.testing.assert_array_equal(xs[:M].cpu().numpy(), xsc)
    wc, wsr = oracle.quantize_rows_fp8(inp["w_gate_up"].reshape(E * 2 * I, H_).float().cpu().numpy())
    np.testing.assert_array_equal(wq.reshape(E * 2 * I, H_).cpu().numpy(), _e4m3_bytes(wc))
    wc, wsr = wc.reshape(E, 2 * I, H_), wsr.reshape(E, 2 * I)
    h_gpu = H.f64(h[:M])
    h_ref = np.zeros((M, I))
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 > r0:
            h_ref[r0:r1] = oracle.expert_gate_up_fp8(xc[r0:r1], xsc[r0:r1], wc[e], wsr[e])
    # h is rounded once to bf16: half an ulp (2^-9 relative) plus fp32 accumulation
    assert (np.abs(h_gpu - h_ref) <= 2.0 ** -8 * np.abs(h_ref) + 1e-4).all()
    # and FP8 stays close to the bf16 gate/up (E4M3 keeps 3 mantissa bits)
    h_bf16 = np.zeros((M, I))
    xp = H.f64(x_perm[:M])
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 > r0:
            h_bf16[r0:r1] = oracle.expert_gate_up(xp[r0:r1], H.f64(inp["w_gate_up"][e]))
    rel = np.linalg.norm(h_gpu - h_bf16) / max(np.linalg.norm(h_bf16), 1e-30)
    assert rel < 0.1


FP8_DOWN_CASES = [
    # T, H, E, K, I, skew   (I % 128 == 0: the down projection's reduction is I)
    (300, 256, 8, 2, 128, "none"), (1000, 512, 64, 4, 256, "normal"), (129, 384, 16, 8, 384, "empties"),
    (64, 256, 16, 8, 128, "normal"), (8, 512, 32, 4, 128, "none"), (1, 256, 8, 2, 128, "none"),
]


@pytest.mark.parametrize("T,H_,E,K,I,skew", FP8_DOWN_CASES)
def test_down_fp8_equals_oracle(moe, T, H_, E, K, I, skew):
    """E4M3 h rows and W_d output channels with per-row scales, quantised on the GPU
    (bit-exact against the oracle), then the FP8 down projection against the oracle's on
    the same codes (fp32 accumulation of exact products)."""
    shape, inp, offsets, _, M = _ffn_inputs(T, H_, E, K, I, "bf16", skew)
    c = _cfg(moe, T, H_, E, K, I=I, dtype="bf16")
    ws = torch.empty(moe.workspace_size(c), dtype=torch.uint8, device="cuda")
    gen = torch.Generator().manual_seed(T + I)
    h = torch.zeros(T * K, I, dtype=torch.bfloat16, device="cuda")
    h[:M] = (torch.randn(M, I, generator=gen) * 0.05).to(torch.bfloat16).cuda()
    hq = torch.empty(T * K, I, dtype=torch.uint8, device="cuda")
    hs = torch.empty(T * K, dtype=torch.float32, device="cuda")
    moe.quantize_fp8(h, hq, hs)
    wq = torch.empty(E, H_, I, dtype=torch.uint8, device="cuda")
    wsc = torch.empty(E, H_, dtype=torch.float32, device="cuda")
    moe.quantize_fp8(inp["w_down"].reshape(E * H_, I), wq, wsc)
    out = torch.full((T * K, H_), -5.0, dtype=torch.float32, device="cuda")
    moe.expert_down_fp8(c, hq, hs, torch.from_numpy(offsets).cuda(), wq, wsc, out, ws)
    torch.cuda.synchronize()
    moe.sync_check()
    assert (out[M:] == -5.0).all()
    hc, hsc = oracle.quantize_rows_fp8(h[:M].float().cpu().numpy())
    np.testing.assert_array_equal(hq[:M].cpu().numpy(), _e4m3_bytes(hc))
    np.testing.assert_array_equal(hs[:M].cpu().numpy(), hsc)
    wc, wsr = oracle.quantize_rows_fp8(inp["w_down"].reshape(E * H_, I).float().cpu().numpy())
    wc, wsr = wc.reshape(E, H_, I), wsr.reshape(E, H_)
    o_ref = np.zeros((M, H_))
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 > r0:
            o_ref[r0:r1] = oracle.expert_down_fp8(hc[r0:r1], hsc[r0:r1], wc[e], wsr[e])
    H.assert_close_y(out[:M].double().cpu().numpy(), o_ref, max_abs=1e-4, rel_l2=1e-5,
                     what="down_fp8")


@pytest.mark.parametrize("H_,I", [(256, 128), (512, 256)])
def test_pair_tiles_fp8(moe, H_, I):
    """The FP8 gate/up and down projection on CTA pairs (groups of >= 384 / 768 rows on
    average), with every kind of last tile (PAIR_GROUPS), against the oracle."""
    sizes = np.array(PAIR_GROUPS)
    E, K = len(sizes), 2
    M = int(sizes.sum())
    T = (M + 255) // K
    offsets = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    shape = synth.MoEShape("pair8", T=T, H=H_, E=E, K=K, I=I, seed=14)
    inp = synth.make_inputs(shape, device="cuda")
    gen = torch.Generator().manual_seed(15)
    x_perm = torch.zeros((T * K, H_), dtype=torch.bfloat16, device="cuda")
    x_perm[:M] = torch.randn(M, H_, generator=gen).to(torch.bfloat16).cuda()
    c = _cfg(moe, T, H_, E, K, I=I, dtype="bf16")
    off = torch.from_numpy(offsets).cuda()
    ws = torch.empty(moe.workspace_size(c), dtype=torch.uint8, device="cuda")
    xq = torch.empty(T * K, H_, dtype=torch.uint8, device="cuda")
    xs = torch.empty(T * K, dtype=torch.float32, device="cuda")
    moe.quantize_fp8(x_perm, xq, xs)
    xq[M:] = 0x7f  # NaN codes after the groups: a leak into a stored row would show
    wgq = torch.empty(E, 2 * I, H_, dtype=torch.uint8, device="cuda")
    wgs = torch.empty(E, 2 * I, dtype=torch.float32, device="cuda")
    moe.quantize_fp8(inp["w_gate_up"].reshape(E * 2 * I, H_), wgq, wgs)
    h = torch.full((T * K, I), -5.0, dtype=torch.bfloat16, device="cuda")
    moe.expert_gate_up_fp8(c, xq, xs, off, wgq, wgs, h, ws)
    hq = torch.empty(T * K, I, dtype=torch.uint8, device="cuda")
    hs = torch.empty(T * K, dtype=torch.float32, device="cuda")
    moe.quantize_fp8(h, hq, hs)
    hq[M:] = 0x7f
    wdq = torch.empty(E, H_, I, dtype=torch.uint8, device="cuda")
    wds = torch.empty(E, H_, dtype=torch.float32, device="cuda")
    moe.quantize_fp8(inp["w_down"].reshape(E * H_, I), wdq, wds)
    out = torch.full((T * K, H_), -5.0, dtype=torch.float32, device="cuda")
    moe.expert_down_fp8(c, hq, hs, off, wdq, wds, out, ws)
    torch.cuda.synchronize()
    moe.sync_check()
    assert (h[M:] == -5.0).all() and (out[M:] == -5.0).all()
    xc, xsc = oracle.quantize_rows_fp8(x_perm[:M].float().cpu().numpy())
    wgc, wgsr = oracle.quantize_rows_fp8(inp["w_gate_up"].reshape(E * 2 * I, H_).float().cpu().numpy())
    wdc, wdsr = oracle.quantize_rows_fp8(inp["w_down"].reshape(E * H_, I).float().cpu().numpy())
    wgc, wgsr = wgc.reshape(E, 2 * I, H_), wgsr.reshape(E, 2 * I)
    wdc, wdsr = wdc.reshape(E, H_, I), wdsr.reshape(E, H_)
    h_gpu = H.f64(h[:M])
    hc, hsc = oracle.quantize_rows_fp8(h[:M].float().cpu().numpy())  # the GPU's h, as the GPU
    o_gpu = out[:M].double().cpu().numpy()
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 == r0:
            continue
        h_ref = oracle.expert_gate_up_fp8(xc[r0:r1], xsc[r0:r1], wgc[e], wgsr[e])
        assert (np.abs(h_gpu[r0:r1] - h_ref) <= 2.0 ** -8 * np.abs(h_ref) + 1e-4).all()
        o_ref = oracle.expert_down_fp8(hc[r0:r1], hsc[r0:r1], wdc[e], wdsr[e])
        H.assert_close_y(o_gpu[r0:r1], o_ref, max_abs=1e-4, rel_l2=1e-5, what="down_fp8")


@pytest.mark.parametrize("T,H_,E,K,I,dtype,skew", [c for c in FFN_CASES if c[5] == "bf16"])
def test_gate_up_row_gather_equals_permuted_copy(moe, T, H_, E, K, I, dtype, skew):
    """The gate/up GEMM that gathers its rows from x by perm computes, row for row, the
    same h as the one reading the permuted copy x_perm (the same products in the same
    order), and reads no entry of perm at or past offsets[E]."""
    shape, inp, offsets, x_perm, M = _ffn_inputs(T, H_, E, K, I, dtype, skew)
    _, _, perm, _ = oracle.permute(_skewed_ids(T, E, K, 0.0, skew, seed=1 + T)[0], E)
    c = _cfg(moe, T, H_, E, K, I=I, dtype=dtype)
    off = torch.from_numpy(offsets).cuda()
    perm_d = torch.full((T * K,), -7, dtype=torch.int32)
    perm_d[:M] = torch.from_numpy(perm[:M])
    perm_d = perm_d.cuda()
    ws = torch.empty(moe.workspace_size(c), dtype=torch.uint8, device="cuda")
    h_copy = torch.full((T * K, I), -5.0, dtype=shape.torch_dtype, device="cuda")
    h_gath = torch.full((T * K, I), -5.0, dtype=shape.torch_dtype, device="cuda")
    moe.expert_gate_up(c, x_perm, off, inp["w_gate_up"], h_copy, ws)
    moe.expert_gate_up_gather(c, inp["x"], perm_d, off, inp["w_gate_up"], h_gath, ws)
    torch.cuda.synchronize()
    assert torch.equal(h_gath[:M], h_copy[:M])
    assert (h_gath[M:] == -5.0).all()


@pytest.mark.parametrize("T,H_,E,K,shared,dtype", [
    (1, 64, 4, 2, False, "bf16"), (300, 256, 8, 2, True, "bf16"), (1000, 512, 128, 8, False, "bf16"),
    (257, 128, 16, 16, True, "f32"), (64, 7168, 256, 8, True, "bf16"),
])
def test_combine(moe, T, H_, E, K, shared, dtype):
    ids, w = _skewed_ids(T, E, K, 0.05, "normal", seed=9)
    _, offsets, perm, inv = oracle.permute(ids, E)
    M = int(offsets[-1])
    g = torch.Generator().manual_seed(3)
    out_perm = torch.randn(T * K, H_, generator=g)
    s = torch.randn(T, H_, generator=g) if shared else None
    c = _cfg(moe, T, H_, E, K, theta=0.05, dtype=dtype)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    y = torch.empty(T, H_, dtype=tdt, device="cuda")
    y32 = torch.empty(T, H_, dtype=torch.float32, device="cuda")
    moe.combine(c, out_perm.cuda(), torch.from_numpy(inv).cuda(), torch.from_numpy(w.astype(np.float32)).cuda(),
                s.cuda() if shared else None, y, y32)
    torch.cuda.synchronize()
    ref = oracle.combine(out_perm.double().numpy()[:M], inv, w.astype(np.float32),
                         s.double().numpy() if shared else None)
    H.assert_close_y(y32.double().cpu().numpy(), ref, max_abs=1e-5, rel_l2=1e-6, what="combine")
    assert torch.equal(y, y32.to(tdt))


CLUSTER_CASES = [
    # T, H, E, K, theta, bias, dup   (bf16, T <= 64, E <= 256: one cluster launch)
    (1, 2048, 128, 8, 0.0, "normal", False),
    (64, 2048, 128, 8, 0.0, "normal", False),
    (33, 256, 40, 6, 0.1, "normal", False),    # E not a multiple of 16; 4 k-blocks, most CTAs none
    (17, 1024, 256, 16, 0.05, "zipf", False),  # two 128-expert tiles, K = 16, gate drop
    (64, 7168, 256, 8, 0.05, "zipf", False),   # 7 k-blocks per CTA through the stage ring
    (8, 64, 8, 2, 0.0, "none", False),         # one k-block for the whole cluster
    (48, 512, 96, 8, 0.0, "none", True),       # exact ties between duplicated experts
    # up to 4 tokens the logits are split by expert over the cluster's CTAs
    (4, 7168, 256, 8, 0.05, "zipf", False),    # 16 experts per CTA, 28 row units per lane
    (4, 320, 40, 6, 0.1, "normal", False),     # ragged units per lane; 2-3 experts per CTA
    (4, 512, 96, 8, 0.0, "none", True),        # exact ties between duplicated experts
    (2, 2048, 128, 8, 0.0, "normal", False),
    (3, 1024, 64, 4, 0.0, "zipf", False),      # padded to 4 tokens; 4 experts per CTA
    (2, 64, 8, 2, 0.0, "none", False),         # fewer experts than CTAs: some have none
    (5, 2048, 128, 8, 0.0, "normal", False),   # the first H-split size
]


@pytest.mark.parametrize("T,H_,E,K,theta,bias,dup", CLUSTER_CASES)
def test_cluster_route_and_dispatch(moe, T, H_, E, K, theta, bias, dup):
    """Decode-sized bf16 batches route and dispatch in one cluster launch.  Its logits match
    the oracle's within fp32 accumulation error; given those logits, its ids and gates equal
    the warp top-k's (moe_route from logits) bit for bit; counts, offsets, perm and inv
    equal moe_permute's on the same ids bit for bit; and the layer output, whose gate/up
    GEMM gathers token rows through perm, matches the oracle."""
    shape = synth.MoEShape("c", T=T, H=H_, E=E, K=K, I=64, theta=theta, dtype="bf16", bias=bias,
                           seed=21)
    inp = synth.make_inputs(shape, device="cuda")
    if dup:
        inp["w_router"][1::2] = inp["w_router"][0::2][: inp["w_router"][1::2].shape[0]]
    run = H.LayerRun(moe, shape, inp)
    run.run()
    moe.sync_check()
    r = run.routing()
    b = inp["router_bias"].cpu().numpy() if inp["router_bias"] is not None else None
    L_ref = oracle.router_logits(H.f64(inp["x"]), H.f64(inp["w_router"]), b)
    assert np.abs(r["logits"] - L_ref).max() <= 1e-4 * max(1.0, np.abs(L_ref).max())
    # the top-k taken on the cluster's own logits
    c = _cfg(moe, T, H_, E, K, theta=theta)
    lg = torch.from_numpy(r["logits"]).cuda()
    ids2 = torch.empty(T, K, dtype=torch.int32, device="cuda")
    w2 = torch.empty(T, K, dtype=torch.float32, device="cuda")
    moe.route(c, None, None, None, lg, ids2, w2)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(r["ids"], ids2.cpu().numpy())
    np.testing.assert_array_equal(r["w"], w2.cpu().numpy())
    # the permutation of those ids
    ws = torch.empty(moe.workspace_size(c), dtype=torch.uint8, device="cuda")
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.full((T * K,), -7, dtype=torch.int32, device="cuda")
    inv = torch.empty(T * K, dtype=torch.int32, device="cuda")
    xp = torch.zeros(T * K, H_, dtype=torch.bfloat16, device="cuda")
    moe.permute(c, inp["x"], ids2, counts, offsets, perm, inv, xp, ws)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(r["counts"], counts.cpu().numpy())
    np.testing.assert_array_equal(r["offsets"], offsets.cpu().numpy())
    M = int(r["offsets"][-1])
    np.testing.assert_array_equal(r["perm"][:M], perm.cpu().numpy()[:M])
    np.testing.assert_array_equal(r["inv"].reshape(-1), inv.cpu().numpy())
    # the layer output: the gate/up GEMM gathers each group's rows from x through perm
    ref = oracle.moe_layer(H.f64(inp["x"]), H.f64(inp["w_router"]), H.f64(inp["w_gate_up"]),
                           H.f64(inp["w_down"]), K, theta, b)
    ok = ~H.ambiguous_tokens(ref["logits"], K, theta, ref["w"])
    H.assert_close_y(run.y32.double().cpu().numpy()[ok], ref["y"][ok])
    # the routing against the oracle's, on the oracle's logits
    L32 = L_ref.astype(np.float32)
    ids_ref, w_ref = oracle.route(L32, K, theta)
    amb = H.compare_routing(L32, r["ids"], r["w"], ids_ref, w_ref, K, theta)
    if not dup:  # duplicated experts tie in every token: only validity is checked there
        assert amb.sum() <= max(1, 0.05 * T)
