"""GPU parity of the whole layer (moe_layer_forward) against the CPU oracle.

* Small layers (all oracle stages in full) covering every feature: float32 and bf16,
  tensor-core and SIMT routers, ragged and empty groups, gate drop, shared expert.
* The workloads at their full sizes, in the launch configuration the benchmark times:
  routing of every token, the permutation's invariants at full size, and the output
  of a sample of tokens (including tokens in the largest and the smallest non-empty
  groups) computed token by token by the oracle.
* Determinism (two runs are bitwise equal) and edge cases (T=0, T=1, K=E, one expert
  takes every token, forced-empty experts).

Output tolerance (bf16 layers): max-abs 2e-2 and relative L2 1e-2 on the fp32 sum
y_f32; the bf16 output y equals the round-to-nearest-even of y_f32 bit for bit, and y
itself is within max-abs 2e-2 plus half a bf16 ulp of the oracle (the store's rounding)
and relative L2 1e-2.  Float32 layers: max-abs and relative L2 1e-3.

At full size the sample holds, besides random tokens, the token of the last row of every
non-empty expert's group and of the first and last rows of its last 128- and 256-row
tiles, so every group's tail tile (single-CTA, CTA-pair and swapped tails) is compared
element by element.
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


def _tol(shape):
    if shape.dtype == "f32":
        return dict(max_abs=H.Y32_MAX_ABS, rel_l2=H.Y32_REL_L2)
    return dict(max_abs=H.Y_MAX_ABS, rel_l2=H.Y_REL_L2)


def _bias_np(inp):
    return inp["router_bias"].cpu().numpy() if inp["router_bias"] is not None else None


def _check_dispatch_properties(r, T, K, E):
    """Invariants of the permutation that hold at any size."""
    ids, counts, offsets, perm, inv = r["ids"], r["counts"], r["offsets"], r["perm"], r["inv"]
    kept = ids >= 0
    M = int(kept.sum())
    assert offsets[0] == 0 and offsets[-1] == M and (np.diff(offsets) == counts).all()
    np.testing.assert_array_equal(counts, np.bincount(ids[kept], minlength=E))
    assert (inv[~kept] == -1).all()
    rows = inv[kept]
    assert np.array_equal(np.sort(rows), np.arange(M))
    tok = np.nonzero(kept)[0]
    np.testing.assert_array_equal(perm[rows], tok)
    exp_of_row = np.repeat(np.arange(E), counts)
    np.testing.assert_array_equal(exp_of_row[rows], ids[kept])
    for e in range(E):
        g = perm[offsets[e]:offsets[e + 1]]
        assert (np.diff(g) > 0).all()


SMALL = [
        synth.WORKLOADS["toy"],
        synth.MoEShape("mixtral_small", T=512, H=512, E=8, K=2, I=1024),
        synth.MoEShape("qwen_small", T=1024, H=256, E=128, K=8, I=128, bias="normal"),
        synth.MoEShape("deepseek_small", T=600, H=512, E=64, K=8, I=256, I_shared=256, theta=0.05,
                       bias="zipf"),
        synth.MoEShape("ragged", T=333, H=192, E=24, K=3, I=192, I_shared=64, theta=0.1,
                       bias="normal", seed=4),
        synth.MoEShape("decode_shared", T=16, H=256, E=32, K=8, I=128, I_shared=128,
                       theta=0.05, bias="zipf", seed=5),
        synth.MoEShape("decode_128", T=128, H=512, E=16, K=4, I=192, I_shared=64, bias="normal",
                       seed=6),
        synth.MoEShape("f32_shared", T=100, H=128, E=6, K=2, I=64, I_shared=128, theta=0.2,
                       dtype="f32", bias="normal", seed=2),
        # decode-sized batches (one-cluster routing, swapped GEMMs): every token-tile width
        # (16, 32, 64), a row gather and a copy of x, ragged I, a shared expert
        synth.MoEShape("decode_t1_tiny", T=1, H=256, E=8, K=2, I=64, seed=7),
        synth.MoEShape("decode_t3_ragged", T=3, H=1024, E=16, K=4, I=320, bias="normal", seed=8),
        synth.MoEShape("decode_t24", T=24, H=512, E=32, K=8, I=192, theta=0.05, bias="zipf",
                       seed=10),
        synth.MoEShape("decode_t64", T=64, H=2048, E=64, K=4, I=128, I_shared=64, bias="normal",
                       seed=11),
]


@pytest.mark.parametrize("fused", [False, True], ids=["gather_combine", "fused_combine"])
@pytest.mark.parametrize("shape", SMALL, ids=lambda s: s.name)
def test_layer_small_full_oracle(moe, shape, fused):
    inp = synth.make_inputs(shape, device="cuda")
    run = H.LayerRun(moe, shape, inp, flags=moe.FLAG_FUSED_COMBINE if fused else 0)
    run.run()
    moe.sync_check()
    r = run.routing()
    f = H.f64
    sh = (f(inp["w_shared_gate_up"]), f(inp["w_shared_down"])) if shape.I_shared else (None, None)
    ref = oracle.moe_layer(f(inp["x"]), f(inp["w_router"]), f(inp["w_gate_up"]), f(inp["w_down"]),
                           shape.K, shape.theta, _bias_np(inp), *sh)
    assert np.abs(r["logits"] - ref["logits"]).max() <= 1e-4 * max(1, np.abs(ref["logits"]).max())
    amb = H.compare_routing(ref["logits"], r["ids"], r["w"], ref["ids"], ref["w"], shape.K, shape.theta)
    _check_dispatch_properties(r, shape.T, shape.K, shape.E)
    if not amb.any():
        np.testing.assert_array_equal(r["counts"], ref["counts"])
        np.testing.assert_array_equal(r["offsets"], ref["offsets"])
        np.testing.assert_array_equal(r["perm"][:len(ref["perm"])], ref["perm"])
        np.testing.assert_array_equal(r["inv"], ref["inv"])
    ok = ~amb
    y32 = run.y32.double().cpu().numpy()
    H.assert_close_y(y32[ok], ref["y"][ok], **_tol(shape))
    assert torch.equal(run.y, run.y32.to(shape.torch_dtype))
    if shape.dtype == "bf16":
        H.assert_close_y_rounded(run.y.double().cpu().numpy()[ok], ref["y"][ok])


def _sample_tokens(r, T, n, seed=0, tails=False):
    """n random tokens plus tokens routed to the largest and smallest groups; with
    `tails`, also the tokens of every non-empty group's last row and of the first and last
    rows of its last 128- and 256-row tiles (the single-CTA and CTA-pair tail tiles)."""
    rng = np.random.default_rng(seed)
    counts, ids = r["counts"], r["ids"]
    nz = np.nonzero(counts)[0]
    big, small = nz[np.argmax(counts[nz])], nz[np.argmin(counts[nz])]
    pick = set(rng.choice(T, size=min(T, n), replace=False).tolist())
    for e in (big, small):
        hit = np.nonzero((ids == e).any(axis=1))[0]
        pick.update(hit[:2].tolist())
    if tails:
        pick.update(_tail_tile_tokens(r).tolist())
    return np.array(sorted(pick))


def _tail_tile_tokens(r):
    """Tokens of every non-empty group's last row and of the first and last rows of its
    last 128- and 256-row tiles."""
    counts, offsets, perm = r["counts"], r["offsets"], r["perm"]
    rows = set()
    for e in np.nonzero(counts)[0]:
        c, o = int(counts[e]), int(offsets[e])
        rows.add(o + c - 1)
        for tile in (128, 256):
            rows.add(o + ((c - 1) // tile) * tile)
            if c > tile:
                rows.add(o + ((c - 1) // tile) * tile - 1)   # last row of the last full tile
    return np.unique(perm[np.array(sorted(rows), dtype=np.int64)])


FULL = [
    ("mixtral", None, 48), ("qwen_prefill", None, 48), ("qwen_decode", 1, 1),
    ("qwen_decode", 8, 8), ("qwen_decode", 32, 32), ("qwen_decode", 64, 64), ("deepseek", None, 24),
    # decode-sized batches of the other two layer shapes: one-cluster routing and swapped
    # GEMMs with H = 4096 and I = 14336 (Mixtral), and with H = 7168, 256 experts, the
    # gate drop and the shared expert (DeepSeek)
    ("mixtral", 4, 4), ("deepseek", 8, 8),
]


@pytest.mark.parametrize("fused", [False, True], ids=["gather_combine", "fused_combine"])
@pytest.mark.parametrize("name,T,nsample", FULL, ids=[f"{n}-{t}" for n, t, _ in FULL])
def test_layer_full_size_sampled(moe, name, T, nsample, fused):
    shape = synth.WORKLOADS[name]
    inp = synth.make_inputs(shape, device="cuda", T=T)
    run = H.LayerRun(moe, shape, inp, flags=moe.FLAG_FUSED_COMBINE if fused else 0)
    run.run()
    moe.sync_check()
    Tn = run.T
    r = run.routing()
    bias = _bias_np(inp)
    x64 = H.f64(inp["x"])
    L_ref = oracle.router_logits(x64, H.f64(inp["w_router"]), bias)
    assert np.abs(r["logits"] - L_ref).max() <= 1e-4 * max(1, np.abs(L_ref).max())
    L32 = L_ref.astype(np.float32)
    ids_ref, w_ref = oracle.route(L32, shape.K, shape.theta)
    amb = H.compare_routing(L32, r["ids"], r["w"], ids_ref, w_ref, shape.K, shape.theta)
    assert amb.mean() < 0.02
    _check_dispatch_properties(r, Tn, shape.K, shape.E)
    if not amb.any():
        _, offsets_ref, _, _ = oracle.permute(ids_ref, shape.E)
        np.testing.assert_array_equal(r["offsets"], offsets_ref)
    toks = _sample_tokens(r, Tn, nsample, tails=True)
    toks = toks[~amb[toks]]
    assert len(toks) >= max(1, nsample // 2), "too few unambiguous sampled tokens"
    # every touched expert's tail tile is in the sample (ambiguous tokens aside)
    checked = set(np.unique(r["ids"][toks][r["ids"][toks] >= 0]).tolist())
    tail_rows = r["offsets"][1:][r["counts"] > 0] - 1
    tail_tok = r["perm"][tail_rows]
    missing = [e for e, t in zip(np.nonzero(r["counts"])[0], tail_tok)
               if not amb[t] and int(e) not in checked]
    assert not missing, f"experts whose tail row was not compared: {missing[:8]}"
    sh = {}
    if shape.I_shared:
        sh = dict(w_shared_gate_up=H.f64(inp["w_shared_gate_up"]), w_shared_down=H.f64(inp["w_shared_down"]))
    ref = oracle.moe_layer_tokens(x64[toks], H.f64(inp["w_router"]), H.ExpertSlices(inp["w_gate_up"]),
                                  H.ExpertSlices(inp["w_down"]), shape.K, shape.theta, bias, **sh)
    np.testing.assert_array_equal(ref["ids"], r["ids"][toks])
    y32 = run.y32.double().cpu().numpy()[toks]
    H.assert_close_y(y32, ref["y"], **_tol(shape))
    assert torch.equal(run.y, run.y32.to(shape.torch_dtype))
    H.assert_close_y_rounded(run.y.double().cpu().numpy()[toks], ref["y"])


def test_fused_combine_matches_gather_combine(moe):
    """The fused combine differs from the deterministic gather only by fp32 rounding order."""
    shape = synth.MoEShape("fc", T=1500, H=512, E=64, K=8, I=256, I_shared=128, theta=0.05,
                           bias="zipf", seed=9)
    inp = synth.make_inputs(shape, device="cuda")
    a = H.LayerRun(moe, shape, inp)
    b = H.LayerRun(moe, shape, inp, flags=moe.FLAG_FUSED_COMBINE)
    a.run()
    b.run()
    torch.cuda.synchronize()
    d = (a.y32 - b.y32).abs().max().item()
    assert d <= 1e-5 * max(1.0, a.y32.abs().max().item())
    assert torch.equal(b.y, b.y32.to(torch.bfloat16))


def test_deterministic(moe):
    shape = synth.MoEShape("det", T=2048, H=512, E=64, K=8, I=256, I_shared=128, theta=0.05,
                           bias="zipf")
    inp = synth.make_inputs(shape, device="cuda")
    a = H.LayerRun(moe, shape, inp)
    b = H.LayerRun(moe, shape, inp)
    a.run()
    b.run()
    a.run()
    torch.cuda.synchronize()
    assert torch.equal(a.y, b.y) and torch.equal(a.y32, b.y32)


@pytest.mark.parametrize("T", [1, 8, 64])
def test_deterministic_decode(moe, T):
    """Decode-sized layers (one-cluster routing, swapped GEMMs) are bitwise repeatable."""
    shape = synth.WORKLOADS["qwen_decode"]
    inp = synth.make_inputs(shape, device="cuda", T=T)
    for flags in (0, moe.FLAG_FUSED_COMBINE):
        a = H.LayerRun(moe, shape, inp, flags=flags)
        b = H.LayerRun(moe, shape, inp, flags=flags)
        a.run()
        b.run()
        a.run()
        torch.cuda.synchronize()
        moe.sync_check()
        if flags == 0:
            assert torch.equal(a.y, b.y) and torch.equal(a.y32, b.y32)
        else:  # the fused combine adds rows at L2 in no fixed order
            assert (a.y32 - b.y32).abs().max().item() <= 1e-5 * max(1.0, a.y32.abs().max().item())


@pytest.mark.parametrize("shape", [
    synth.MoEShape("cap_qwen_small", T=1024, H=256, E=128, K=8, I=128, bias="normal", seed=21),
    # no gate drop here: with it, one near-threshold gate decided differently from the
    # layer's own logits would reroute later tokens (the route-level capacity tests cover
    # the drop, on given logits with every gate clear of the threshold)
    synth.MoEShape("cap_shared_zipf", T=600, H=512, E=64, K=8, I=256, I_shared=256,
                   bias="zipf", seed=22),
    synth.MoEShape("cap_decode", T=8, H=512, E=32, K=4, I=128, bias="zipf", seed=23),
], ids=lambda s: s.name)
def test_layer_with_capacity_routing(moe, shape):
    """MOE_FLAG_CAPACITY through the whole layer.  The oracle routes from the layer's own
    fp32 logits (checked against the oracle's separately), so both take the same integer
    decisions; the rest of the layer is compared within the usual tolerance."""
    inp = synth.make_inputs(shape, device="cuda")
    run = H.LayerRun(moe, shape, inp, flags=moe.FLAG_CAPACITY)
    run.run()
    torch.cuda.synchronize()
    moe.sync_check()
    r = run.routing()
    bias = _bias_np(inp)
    x64 = H.f64(inp["x"])
    L_ref = oracle.router_logits(x64, H.f64(inp["w_router"]), bias)
    assert np.abs(r["logits"] - L_ref).max() <= 1e-4 * max(1, np.abs(L_ref).max())
    L32 = r["logits"].astype(np.float32)
    ids_ref, w_ref = oracle.route_capacity(L32, shape.K, shape.theta)
    assert H.capacity_gate_margin(L32, shape.K, shape.theta, ids_ref) > 1e-5
    np.testing.assert_array_equal(r["ids"], ids_ref)
    np.testing.assert_allclose(r["w"], w_ref, rtol=0, atol=1e-5)
    counts_ref, offsets_ref, perm_ref, inv_ref = oracle.permute(ids_ref, shape.E)
    assert counts_ref.max() <= oracle.capacity(shape.T, shape.K, shape.E)
    np.testing.assert_array_equal(r["offsets"], offsets_ref)
    out_ref = oracle.grouped_ffn(x64[perm_ref], offsets_ref, H.ExpertSlices(inp["w_gate_up"]),
                                 H.ExpertSlices(inp["w_down"]))
    shared_ref = None
    if shape.I_shared:
        shared_ref = oracle.swiglu_ffn(x64, H.f64(inp["w_shared_gate_up"]),
                                       H.f64(inp["w_shared_down"]))
    y_ref = oracle.combine(out_ref, inv_ref, w_ref, shared_ref)
    H.assert_close_y(run.y32.double().cpu().numpy(), y_ref, **_tol(shape))
    assert torch.equal(run.y, run.y32.to(shape.torch_dtype))


@pytest.mark.parametrize("shape", [
    synth.MoEShape("fp8_prefill", T=300, H=256, E=8, K=2, I=128, seed=31),
    synth.MoEShape("fp8_shared", T=129, H=384, E=16, K=8, I=256, I_shared=128, bias="normal",
                   seed=32),
    synth.MoEShape("fp8_decode", T=8, H=512, E=32, K=4, I=128, bias="zipf", seed=33),
], ids=lambda s: s.name)
@pytest.mark.parametrize("fused", [False, True], ids=["gather_combine", "fused_combine"])
def test_layer_fp8_equals_oracle(moe, shape, fused):
    """moe_layer_forward_fp8: E4M3 experts (weights per output channel, x and h per row)
    against the oracle's FP8 expert chain.  The oracle routes from the layer's own fp32
    logits; h is the oracle's (fp64, rounded once to bf16), so a rare one-ulp difference of
    h can move one E4M3 code: the output is compared within the layer tolerance."""
    T, H_, E, K, I = shape.T, shape.H, shape.E, shape.K, shape.I
    inp = synth.make_inputs(shape, device="cuda")
    cfg = moe.MoEConfig.make(T, H_, E, K, I, shape.I_shared, shape.theta, moe.BF16,
                             moe.FLAG_FP8 | (moe.FLAG_FUSED_COMBINE if fused else 0))
    ws = torch.empty(moe.workspace_size(cfg), dtype=torch.uint8, device="cuda")
    wgq = torch.empty(E, 2 * I, H_, dtype=torch.uint8, device="cuda")
    wgs = torch.empty(E, 2 * I, dtype=torch.float32, device="cuda")
    moe.quantize_fp8(inp["w_gate_up"].reshape(E * 2 * I, H_), wgq, wgs)
    wdq = torch.empty(E, H_, I, dtype=torch.uint8, device="cuda")
    wds = torch.empty(E, H_, dtype=torch.float32, device="cuda")
    moe.quantize_fp8(inp["w_down"].reshape(E * H_, I), wdq, wds)
    y = torch.empty(T, H_, dtype=torch.bfloat16, device="cuda")
    y32 = torch.empty(T, H_, dtype=torch.float32, device="cuda")
    moe.layer_forward_fp8(cfg, inp["x"], inp["w_router"], inp["router_bias"], wgq, wgs, wdq, wds,
                          inp.get("w_shared_gate_up"), inp.get("w_shared_down"), y, y32, ws)
    torch.cuda.synchronize()
    moe.sync_check()
    run = H.LayerRun(moe, shape, inp)  # only for its workspace views
    run.cfg, run.ws = cfg, ws
    r = run.routing()
    x64 = H.f64(inp["x"])
    L_ref = oracle.router_logits(x64, H.f64(inp["w_router"]), _bias_np(inp))
    assert np.abs(r["logits"] - L_ref).max() <= 1e-4 * max(1, np.abs(L_ref).max())
    ids_ref, w_ref = oracle.route(r["logits"].astype(np.float32), K, shape.theta)
    np.testing.assert_array_equal(r["ids"], ids_ref)
    counts_ref, offsets_ref, perm_ref, inv_ref = oracle.permute(ids_ref, E)
    np.testing.assert_array_equal(r["offsets"], offsets_ref)
    xc, xs = oracle.quantize_rows_fp8(inp["x"].float().cpu().numpy())
    wgc, wgsr = oracle.quantize_rows_fp8(inp["w_gate_up"].reshape(E * 2 * I, H_).float().cpu().numpy())
    wdc, wdsr = oracle.quantize_rows_fp8(inp["w_down"].reshape(E * H_, I).float().cpu().numpy())
    wgc, wgsr = wgc.reshape(E, 2 * I, H_), wgsr.reshape(E, 2 * I)
    wdc, wdsr = wdc.reshape(E, H_, I), wdsr.reshape(E, H_)
    M = int(offsets_ref[-1])
    o_ref = np.zeros((M, H_))
    for e in range(E):
        r0, r1 = int(offsets_ref[e]), int(offsets_ref[e + 1])
        if r1 == r0:
            continue
        rows = perm_ref[r0:r1]
        h = oracle.expert_gate_up_fp8(xc[rows], xs[rows], wgc[e], wgsr[e])
        h = torch.from_numpy(h).to(torch.bfloat16).float().numpy()  # rounded once to bf16
        hc, hsc = oracle.quantize_rows_fp8(h)
        o_ref[r0:r1] = oracle.expert_down_fp8(hc, hsc, wdc[e], wdsr[e])
    shared_ref = None
    if shape.I_shared:
        shared_ref = oracle.swiglu_ffn(x64, H.f64(inp["w_shared_gate_up"]),
                                       H.f64(inp["w_shared_down"]))
    y_ref = oracle.combine(o_ref, inv_ref, w_ref, shared_ref)
    H.assert_close_y(y32.double().cpu().numpy(), y_ref, **_tol(shape))
    assert torch.equal(y, y32.to(torch.bfloat16))


@pytest.mark.parametrize("case", ["T0", "T1", "K_eq_E", "one_expert", "empty_experts"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_edge_cases(moe, case, dtype):
    base = dict(T=300, H=128, E=8, K=2, I=128, dtype=dtype, seed=8)
    if case == "T0":
        base["T"] = 0
    elif case == "T1":
        base["T"] = 1
    elif case == "K_eq_E":
        base.update(E=4, K=4)
    shape = synth.MoEShape(case, **base)
    inp = synth.make_inputs(shape, device="cuda")
    if case == "one_expert":
        inp["router_bias"] = torch.full((shape.E,), -1e4, device="cuda")
        inp["router_bias"][5] = 0.0
        inp["router_bias"][2] = 0.0
    elif case == "empty_experts":
        inp["router_bias"] = torch.zeros(shape.E, device="cuda")
        inp["router_bias"][1::2] = -1e4
    run = H.LayerRun(moe, shape, inp)
    run.run()
    moe.sync_check()
    if shape.T == 0:
        return
    r = run.routing()
    f = H.f64
    ref = oracle.moe_layer(f(inp["x"]), f(inp["w_router"]), f(inp["w_gate_up"]), f(inp["w_down"]),
                           shape.K, shape.theta, _bias_np(inp))
    amb = H.compare_routing(ref["logits"], r["ids"], r["w"], ref["ids"], ref["w"], shape.K, shape.theta)
    if case in ("one_expert", "empty_experts"):
        assert not amb.any()
        np.testing.assert_array_equal(r["counts"], ref["counts"])
        if case == "empty_experts":
            assert (r["counts"][1::2] == 0).all()
        else:
            assert set(np.nonzero(r["counts"])[0]) == {2, 5}
    H.assert_close_y(run.y32.double().cpu().numpy()[~amb], ref["y"][~amb], **_tol(shape))


def test_streams_and_sync_check(moe):
    shape = synth.MoEShape("s", T=512, H=256, E=16, K=4, I=128, bias="normal")
    inp = synth.make_inputs(shape, device="cuda")
    s = torch.cuda.Stream()
    a = H.LayerRun(moe, shape, inp)
    with torch.cuda.stream(s):
        a.run(stream=s)
    moe.sync_check(s)
    b = H.LayerRun(moe, shape, inp)
    b.run()
    torch.cuda.synchronize()
    assert torch.equal(a.y, b.y)


def test_kernel_launch_counter(moe):
    """moe_kernel_launch_count() grows by the same number for two identical layer calls,
    by at least one launch per stage, and not at all for an empty batch."""
    shape = synth.MoEShape("cnt", T=700, H=256, E=32, K=4, I=128, I_shared=64, bias="normal",
                           seed=12)
    inp = synth.make_inputs(shape, device="cuda")
    run = H.LayerRun(moe, shape, inp)
    deltas = []
    for _ in range(2):
        n0 = moe.kernel_launch_count()
        run.run()
        deltas.append(moe.kernel_launch_count() - n0)
    moe.sync_check()
    assert deltas[0] == deltas[1] >= 5      # route, permute, gate/up, down, combine at least
    empty = H.LayerRun(moe, shape, {k: v[:0] if k == "x" else v for k, v in inp.items()}, T=0)
    n0 = moe.kernel_launch_count()
    empty.run()
    assert moe.kernel_launch_count() == n0


@pytest.mark.parametrize("fused", [False, True], ids=["gather_combine", "fused_combine"])
def test_shared_expert_on_side_stream_matches_in_order_layer(moe, fused):
    """From 1024 tokens the shared expert runs on the library's side stream, concurrently
    with the permutation; under graph capture the layer runs in stream order instead.  Both
    must give the same output (bitwise with the deterministic gather combine)."""
    shape = synth.MoEShape("side", T=2048, H=512, E=64, K=8, I=256, I_shared=256, theta=0.05,
                           bias="zipf", seed=15)
    inp = synth.make_inputs(shape, device="cuda")
    flags = moe.FLAG_FUSED_COMBINE if fused else 0
    eager = H.LayerRun(moe, shape, inp, flags=flags)
    eager.run()
    moe.sync_check()
    cap = H.LayerRun(moe, shape, inp, flags=flags)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cap.run(stream=torch.cuda.current_stream())
    g.replay()
    torch.cuda.synchronize()
    moe.sync_check()
    if fused:   # additions in no fixed order
        torch.testing.assert_close(eager.y32, cap.y32, rtol=1e-5, atol=1e-5)
    else:
        assert torch.equal(eager.y, cap.y) and torch.equal(eager.y32, cap.y32)
    # and against the oracle on a sample of tokens
    r = eager.routing()
    toks = np.arange(0, shape.T, 97)
    sh = dict(w_shared_gate_up=H.f64(inp["w_shared_gate_up"]), w_shared_down=H.f64(inp["w_shared_down"]))
    ref = oracle.moe_layer_tokens(H.f64(inp["x"])[toks], H.f64(inp["w_router"]),
                                  H.ExpertSlices(inp["w_gate_up"]), H.ExpertSlices(inp["w_down"]),
                                  shape.K, shape.theta, _bias_np(inp), **sh)
    L32 = r["logits"][toks]
    amb = H.ambiguous_tokens(L32, shape.K, shape.theta, ref["w"])
    H.assert_close_y(eager.y32.double().cpu().numpy()[toks][~amb], ref["y"][~amb])


@pytest.mark.parametrize("fill", [0x00, 0xFF, 0x7F], ids=["zeros", "ones", "large"])
def test_workspace_contents_do_not_matter(moe, fill):
    """Every workspace field a call reads is written by that call first.  In particular the
    tile counter of the routed gate/up GEMM on CTA pairs (tiles drawn in index order) is
    zeroed by the call's permutation kernel (the layer) or a memset (the standalone call):
    a stale or garbage counter would make the pairs skip tiles.  The layer's shape puts the
    gate/up on CTA pairs (512 rows per expert)."""
    shape = synth.MoEShape("wsfill", T=2048, H=512, E=32, K=8, I=256, I_shared=128, theta=0.0,
                           bias="normal", seed=21)
    inp = synth.make_inputs(shape, device="cuda")
    clean = H.LayerRun(moe, shape, inp)
    clean.ws.zero_()
    clean.run()
    run = H.LayerRun(moe, shape, inp)
    run.ws.fill_(fill)
    run.run()
    run.run()  # and again on the workspace the first call left behind
    moe.sync_check()
    assert torch.equal(run.y, clean.y) and torch.equal(run.y32, clean.y32)
    # the standalone gate/up on the same routing, with a filled workspace
    r = clean.routing()
    T, K = shape.T, shape.K
    x_perm = clean.view("x_perm", (T * K, shape.H), torch.bfloat16).clone()
    offsets = torch.from_numpy(r["offsets"]).cuda()
    h_clean = torch.empty(T * K, shape.I, dtype=torch.bfloat16, device="cuda")
    h_fill = torch.empty_like(h_clean)
    ws2 = torch.full_like(run.ws, fill)
    moe.expert_gate_up(clean.cfg, x_perm, offsets, inp["w_gate_up"], h_clean, clean.ws)
    moe.expert_gate_up(clean.cfg, x_perm, offsets, inp["w_gate_up"], h_fill, ws2)
    moe.sync_check()
    M = int(r["offsets"][-1])
    assert torch.equal(h_fill[:M], h_clean[:M])
    # the FP8 layer, whose permutation zeroes the same counter
    E, I, Hd = shape.E, shape.I, shape.H
    wq = torch.empty(E, 2 * I, Hd, dtype=torch.uint8, device="cuda")
    wsc = torch.empty(E, 2 * I, device="cuda")
    moe.quantize_fp8(inp["w_gate_up"].reshape(E * 2 * I, Hd), wq, wsc)
    wdq = torch.empty(E, Hd, I, dtype=torch.uint8, device="cuda")
    wds = torch.empty(E, Hd, device="cuda")
    moe.quantize_fp8(inp["w_down"].reshape(E * Hd, I), wdq, wds)
    cfg8 = moe.MoEConfig.make(T, Hd, E, K, I, shape.I_shared, shape.theta, moe.BF16, moe.FLAG_FP8)
    outs = []
    for f in (0x00, fill):
        ws8 = torch.full((moe.workspace_size(cfg8),), f, dtype=torch.uint8, device="cuda")
        y8 = torch.empty(T, Hd, dtype=torch.bfloat16, device="cuda")
        moe.layer_forward_fp8(cfg8, inp["x"], inp["w_router"], inp["router_bias"], wq, wsc, wdq,
                              wds, inp["w_shared_gate_up"], inp["w_shared_down"], y8, None, ws8)
        outs.append(y8)
    moe.sync_check()
    assert torch.equal(outs[0], outs[1])


@pytest.mark.parametrize("name", ["qwen_prefill", "mixtral"])
def test_layer_fp8_full_size_sampled(moe, name):
    """moe_layer_forward_fp8 at full size (Qwen3 shape, T=8192: the FP8 gate/up on CTA pairs
    with the dynamic tile order, the FP8 scatter-add down projection with eight epilogue
    warps; Mixtral shape: both FP8 GEMMs on CTA pairs) against the oracle's FP8 expert chain on sampled tokens, every touched expert's
    last row among them.  The oracle quantises the weights of every expert they use itself,
    and routes from the layer's own fp32 logits (as the small FP8 test does)."""
    shape = synth.WORKLOADS[name]
    T, H_, E, K, I = shape.T, shape.H, shape.E, shape.K, shape.I
    inp = synth.make_inputs(shape, device="cuda")
    cfg = moe.MoEConfig.make(T, H_, E, K, I, shape.I_shared, shape.theta, moe.BF16,
                             moe.FLAG_FP8 | moe.FLAG_FUSED_COMBINE)
    ws = torch.empty(moe.workspace_size(cfg), dtype=torch.uint8, device="cuda")
    wgq = torch.empty(E, 2 * I, H_, dtype=torch.uint8, device="cuda")
    wgs = torch.empty(E, 2 * I, dtype=torch.float32, device="cuda")
    moe.quantize_fp8(inp["w_gate_up"].reshape(E * 2 * I, H_), wgq, wgs)
    wdq = torch.empty(E, H_, I, dtype=torch.uint8, device="cuda")
    wds = torch.empty(E, H_, dtype=torch.float32, device="cuda")
    moe.quantize_fp8(inp["w_down"].reshape(E * H_, I), wdq, wds)
    y = torch.empty(T, H_, dtype=torch.bfloat16, device="cuda")
    y32 = torch.empty(T, H_, dtype=torch.float32, device="cuda")
    moe.layer_forward_fp8(cfg, inp["x"], inp["w_router"], inp["router_bias"], wgq, wgs, wdq, wds,
                          inp.get("w_shared_gate_up"), inp.get("w_shared_down"), y, y32, ws)
    torch.cuda.synchronize()
    moe.sync_check()
    run = H.LayerRun(moe, shape, inp)  # only for its workspace views
    run.cfg, run.ws = cfg, ws
    r = run.routing()
    _check_dispatch_properties(r, T, K, E)
    ids_ref, w_ref = oracle.route(r["logits"].astype(np.float32), K, shape.theta)
    np.testing.assert_array_equal(r["ids"], ids_ref)
    toks = _sample_tokens(r, T, 8, tails=True)
    xc, xs = oracle.quantize_rows_fp8(inp["x"][toks].float().cpu().numpy())
    wg_cache, wd_cache = {}, {}

    def expert(e):
        if e not in wg_cache:
            wg_cache[e] = oracle.quantize_rows_fp8(inp["w_gate_up"][e].float().cpu().numpy())
            wd_cache[e] = oracle.quantize_rows_fp8(inp["w_down"][e].float().cpu().numpy())
        return wg_cache[e], wd_cache[e]

    y_ref = np.zeros((len(toks), H_))
    for i, t in enumerate(toks):
        for k in range(K):
            e = int(ids_ref[t, k])
            if e < 0:
                continue
            (wgc, wgsr), (wdc, wdsr) = expert(e)
            h = oracle.expert_gate_up_fp8(xc[i:i + 1], xs[i:i + 1], wgc, wgsr)
            h = torch.from_numpy(h).to(torch.bfloat16).float().numpy()  # rounded once to bf16
            hc, hsc = oracle.quantize_rows_fp8(h)
            y_ref[i] += w_ref[t, k] * oracle.expert_down_fp8(hc, hsc, wdc, wdsr)[0]
    H.assert_close_y(y32.double().cpu().numpy()[toks], y_ref, **_tol(shape))
    assert torch.equal(y, y32.to(torch.bfloat16))
