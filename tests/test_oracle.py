"""Pins of the CPU oracle against facts that do not come from the oracle.

Each test checks one oracle function against an independent statement of the
same result: a hand-worked example (tests/golden/hand_example.json), published
format tables (tests/golden/formats.json), library routines (torch's float8
cast, scipy's softmax, torch's silu), brute force on tiny inputs, closed-form
special cases and invariants.  tests/test_oracle_mutants.py shows that
plausible mistakes in the oracle are caught by these pins.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
import moe_synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as fh:
        return json.load(fh)


def _num(v):
    if isinstance(v, str):
        if v == "ln3":
            return math.log(3.0)
        if v == "-ln3":
            return -math.log(3.0)
        if "/" in v:
            a, b = v.split("/")
            return float(a) / float(b)
    return float(v)


def _arr(nested):
    if isinstance(nested, list):
        return np.array([_arr(v) for v in nested], dtype=np.float64)
    return _num(nested)


class _Inputs:
    """Minimal stand-in for moe_synth.MoEInputs built from a fixture."""

    def __init__(self, cfg, **kw):
        self.cfg = cfg
        self.bias = None
        for n in ("w13_scale", "w13_gscale", "w2_scale", "w2_gscale",
                  "s13_scale", "s13_gscale", "s2_scale", "s2_gscale"):
            setattr(self, n, None)
        for k, v in kw.items():
            setattr(self, k, v)


def hand_inputs():
    g = _load("hand_example.json")
    cfg = moe_synth.MoEConfig("hand", 1, 2, 4, 2, 1, 1, "f32", "f32")
    inp = _Inputs(cfg, x=_arr(g["x"]), w_router=_arr(g["w_router"]), w13=_arr(g["w13"]),
                  w2=_arr(g["w2"]), s13=_arr(g["s13"])[None], s2=_arr(g["s2"])[None])
    return inp, g["expected"]


# ---------------------------------------------------------------- formats

def test_e4m3_table_matches_torch_cast():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = oracle.E4M3_TABLE
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_e4m3_named_codes():
    g = _load("formats.json")
    for code, val in g["e4m3_named_codes"].items():
        got = oracle.E4M3_TABLE[int(code, 16)]
        assert got == val and math.copysign(1, got) == math.copysign(1, val), code
    for code in g["e4m3_nan_codes"]:
        assert math.isnan(oracle.E4M3_TABLE[int(code, 16)])


def test_e2m1_grid():
    g = _load("formats.json")
    mags = np.array(g["e2m1_magnitudes_by_code"])
    assert np.array_equal(oracle.E2M1_TABLE[:8], mags)
    assert np.array_equal(oracle.E2M1_TABLE[8:], -mags)


def test_e2m1_packing_nibble_order():
    # element 2i in the low nibble: byte 0x71 = [code 1, code 7] = [0.5, 6.0]
    v = oracle.decode_e2m1_packed(np.array([[0x71, 0x8F]], dtype=np.uint8))
    assert v.tolist() == [[0.5, 6.0, -6.0, -0.0]]


def test_bf16_decode_matches_torch():
    rng = np.random.default_rng(1)
    a = torch.from_numpy(rng.standard_normal(1000).astype(np.float32) * 100).to(torch.bfloat16)
    bits = a.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.decode_bf16(bits), a.to(torch.float64).numpy())


def test_nvfp4_dequant_nearest_grid_roundtrip():
    # The generator's quantiser picks, per element, the e2m1 grid point nearest
    # to w/(s_b g); the oracle's dequant must reproduce exactly that grid point
    # times the decoded scales (brute force over the 8 magnitudes).
    rng = np.random.default_rng(2)
    w = rng.standard_normal((8, 64)).astype(np.float32) / 8
    packed, bs, g = moe_synth.quantize_nvfp4(w)
    deq = oracle.dequant("nvfp4", packed, bs, g)
    scale = np.repeat(torch.from_numpy(bs).view(torch.float8_e4m3fn).to(torch.float64).numpy(), 16, 1) * float(g)
    grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6], dtype=np.float64)
    v = w.astype(np.float64) / scale
    dist = np.abs(np.abs(v)[..., None] - grid)
    best = grid[np.argmin(dist, axis=-1)] * np.sign(v)
    # exact ties are measure-zero for normal data
    assert np.array_equal(deq, best * scale)


def test_fp8_dequant_matches_torch():
    rng = np.random.default_rng(3)
    w = rng.standard_normal((16, 32)).astype(np.float32)
    q, s = moe_synth.quantize_e4m3_rows(w)
    deq = oracle.dequant("e4m3", q, s)
    ref = torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float64).numpy() * s[:, None]
    assert np.array_equal(deq, ref)
    # per-channel scales: the largest magnitude of each row decodes to 448*s
    assert np.allclose(np.max(np.abs(deq), axis=1), 448 * s.astype(np.float64))


# ---------------------------------------------------------------- hand example

def test_hand_example():
    inp, exp = hand_inputs()
    res = oracle.layer_forward(inp)
    assert res["ids"].tolist() == exp["ids"]
    assert np.allclose(res["w"], _arr(exp["w"]), rtol=0, atol=1e-15)
    assert np.allclose(res["y"] / math.log(3.0), _arr(exp["y_over_ln3"]), rtol=0, atol=1e-13)


def test_hand_example_token_subset_path():
    inp, exp = hand_inputs()
    res = oracle.layer_forward_tokens(inp, [0])
    assert np.allclose(res["y"] / math.log(3.0), _arr(exp["y_over_ln3"]), rtol=0, atol=1e-13)


# ---------------------------------------------------------------- routing

def _brute_rank_ids(L, k):
    """ids by counting, for every expert, how many experts precede it under
    the order (higher logit first, then lower index)."""
    T, E = L.shape
    ids = np.zeros((T, k), dtype=np.int32)
    for t in range(T):
        for e in range(E):
            r = sum(1 for e2 in range(E) if L[t, e2] > L[t, e] or (L[t, e2] == L[t, e] and e2 < e))
            if r < k:
                ids[t, r] = e
    return ids


@pytest.mark.parametrize("E,k", [(8, 1), (8, 3), (8, 8), (16, 6), (128, 6), (128, 8)])
def test_topk_bruteforce_with_exact_ties(E, k):
    rng = np.random.default_rng(E * 10 + k)
    L = rng.integers(-3, 4, size=(40, E)).astype(np.float64)   # many exact ties
    assert np.array_equal(oracle.topk_ids(L, k), _brute_rank_ids(L, k))
    L2 = rng.standard_normal((40, E))
    assert np.array_equal(oracle.topk_ids(L2, k), _brute_rank_ids(L2, k))


def test_topk_subset_maximises_logit_sum():
    # Brute force over all k-subsets on a tiny E: the selected set has the
    # largest sum of logits (distinct logits).
    rng = np.random.default_rng(4)
    E, k = 7, 3
    L = rng.standard_normal((20, E))
    ids = oracle.topk_ids(L, k)
    for t in range(20):
        best = max(itertools.combinations(range(E), k), key=lambda s: sum(L[t, list(s)]))
        assert set(ids[t]) == set(best)


def test_gates_equal_full_softmax_restricted_renormalised():
    rng = np.random.default_rng(5)
    L = rng.standard_normal((50, 128)) * 3
    ids = oracle.topk_ids(L, 6)
    p = scipy.special.softmax(L, axis=1)
    sel = np.take_along_axis(p, ids.astype(np.int64), axis=1)
    ref = sel / sel.sum(axis=1, keepdims=True)
    assert np.allclose(oracle.gates(L, ids), ref, rtol=1e-13, atol=0)


def test_gates_special_cases():
    rng = np.random.default_rng(6)
    L = rng.standard_normal((30, 16)) * 5
    # k = 1: the single gate is exactly one
    assert np.array_equal(oracle.gates(L, oracle.topk_ids(L, 1)), np.ones((30, 1)))
    # k = E: dense softmax mixture (in the selected order)
    ids = oracle.topk_ids(L, 16)
    assert np.allclose(oracle.gates(L, ids),
                       np.take_along_axis(scipy.special.softmax(L, axis=1), ids.astype(np.int64), 1),
                       rtol=1e-13, atol=0)
    # gates descend with the ids order and sum to one
    w = oracle.gates(L, oracle.topk_ids(L, 6))
    assert np.all(np.diff(w, axis=1) <= 0)
    assert np.allclose(w.sum(1), 1.0, rtol=0, atol=1e-15)


def test_router_logits_bias_and_linearity():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((5, 32))
    W = rng.standard_normal((8, 32))
    b = rng.standard_normal(8)
    L = oracle.router_logits(x, W, b)
    ref = torch.nn.functional.linear(torch.from_numpy(x), torch.from_numpy(W), torch.from_numpy(b)).numpy()
    assert np.allclose(L, ref, rtol=1e-13, atol=1e-13)


def test_near_tie_flags():
    L = np.array([[5.0, 4.0, 3.0, 2.99995, 1.0],     # k=3: 3rd vs 4th within 1e-4
                  [5.0, 4.99999, 3.0, 2.0, 1.0],     # order tie inside the top 3
                  [5.0, 4.0, 3.0, 2.0, 1.0]])
    sel, order = oracle.near_ties(L, 3)
    assert sel.tolist() == [True, False, False]
    assert order.tolist() == [False, True, False]


# ---------------------------------------------------------------- permutation

def _brute_permute(ids, E):
    T, k = ids.shape
    sorted_pair = []
    counts = []
    for e in range(E):
        c = 0
        for t in range(T):
            for j in range(k):
                if ids[t, j] == e:
                    sorted_pair.append(t * k + j)
                    c += 1
        counts.append(c)
    return np.array(counts), np.array(sorted_pair)


@pytest.mark.parametrize("T,E,k", [(1, 4, 2), (7, 8, 3), (33, 128, 6), (64, 128, 8)])
def test_permute_bruteforce_and_invariants(T, E, k):
    rng = np.random.default_rng(T + E + k)
    L = rng.standard_normal((T, E))
    ids = oracle.topk_ids(L, k)
    counts, offsets, sp, row_of = oracle.permute(ids, E)
    bc, bsp = _brute_permute(ids, E)
    assert np.array_equal(counts, bc)
    assert np.array_equal(sp, bsp)
    assert offsets[0] == 0 and offsets[-1] == T * k and np.all(np.diff(offsets) == counts)
    assert np.array_equal(np.sort(sp), np.arange(T * k))                     # bijection
    assert np.array_equal(row_of[sp], np.arange(T * k))                      # inverse
    for e in range(E):                                                       # one token once per expert
        toks = sp[offsets[e]:offsets[e + 1]] // k
        assert len(set(toks.tolist())) == len(toks)
        assert np.all(np.diff(toks) > 0)


def test_permute_empty_experts():
    ids = np.array([[0, 1], [1, 0], [3, 1]], dtype=np.int32)
    counts, offsets, sp, row_of = oracle.permute(ids, 5)
    assert counts.tolist() == [2, 3, 0, 1, 0]
    assert offsets.tolist() == [0, 2, 5, 5, 6, 6]
    assert sp.tolist() == [0, 3, 1, 2, 5, 4]


# ---------------------------------------------------------------- FFN / layer

def _torch_swiglu(X, W13, W2):
    X, W13, W2 = (torch.from_numpy(np.asarray(a, np.float64)) for a in (X, W13, W2))
    f = W2.shape[1]
    g, u = torch.nn.functional.linear(X, W13).split(f, dim=-1)
    return torch.nn.functional.linear(torch.nn.functional.silu(g) * u, W2).numpy()


def test_swiglu_matches_torch():
    rng = np.random.default_rng(8)
    X = rng.standard_normal((9, 16))
    W13 = rng.standard_normal((2 * 16, 16)) / 4      # f = d = 16 so a transpose would still run
    W2 = rng.standard_normal((16, 16)) / 4
    assert np.allclose(oracle.swiglu_ffn(X, W13, W2), _torch_swiglu(X, W13, W2), rtol=1e-12, atol=1e-12)


def test_silu_special_values():
    z = np.array([0.0, math.log(3.0), -math.log(3.0), 50.0, -50.0])
    s = oracle.silu(z)
    assert s[0] == 0.0
    assert math.isclose(s[1], 0.75 * math.log(3.0), rel_tol=1e-15)
    assert math.isclose(s[2], -0.25 * math.log(3.0), rel_tol=1e-15)
    assert math.isclose(s[3], 50.0, rel_tol=1e-15) and abs(s[4]) < 1e-19


@pytest.mark.parametrize("w_dtype", ["f32", "e4m3", "nvfp4"])
def test_dense_equivalence(w_dtype):
    """All routed experts identical => y = FFN(x) + shared(x) for any routing,
    because the renormalised gates sum to one."""
    inp = moe_synth.make_custom(T=24, d=64, E=16, k=4, f=32, fs=32, x_dtype="bf16", w_dtype=w_dtype, seed=11)
    for name in ("w13", "w13_scale", "w13_gscale", "w2", "w2_scale", "w2_gscale"):
        a = getattr(inp, name)
        if a is not None:
            a[:] = a[:1]
    res = oracle.layer_forward(inp)
    x = oracle.x_values(inp)
    W13, W2 = oracle.expert_weights(inp, 0)
    S13, S2 = oracle.shared_weights(inp)
    ref = _torch_swiglu(x, W13, W2) + _torch_swiglu(x, S13, S2)
    assert np.allclose(res["y"], ref, rtol=1e-11, atol=1e-12)
    # a router bias changes the routing but not y
    inp.bias = np.linspace(-3, 3, 16).astype(np.float32)
    res2 = oracle.layer_forward(inp)
    assert not np.array_equal(res2["ids"], res["ids"])
    assert np.allclose(res2["y"], ref, rtol=1e-11, atol=1e-12)


def test_layer_equals_per_token_mixture():
    """Brute-force restatement per token: y[t] = shared(x_t) + sum_j w_j FFN_{ids_j}(x_t),
    each expert applied to one token at a time through torch."""
    inp = moe_synth.make_custom(T=6, d=32, E=8, k=3, f=16, fs=8, x_dtype="f32", w_dtype="f32", seed=12)
    res = oracle.layer_forward(inp)
    x = oracle.x_values(inp)
    p = scipy.special.softmax(oracle.router_logits(x, inp.w_router, None), axis=1)
    S13, S2 = oracle.shared_weights(inp)
    for t in range(6):
        top = sorted(range(8), key=lambda e: (-p[t, e], e))[:3]
        wsum = sum(p[t, e] for e in top)
        y = _torch_swiglu(x[t:t + 1], S13, S2)[0]
        for e in top:
            W13, W2 = oracle.expert_weights(inp, e)
            y = y + (p[t, e] / wsum) * _torch_swiglu(x[t:t + 1], W13, W2)[0]
        assert np.allclose(res["y"][t], y, rtol=1e-12, atol=1e-12)


def test_token_subset_matches_full():
    inp = moe_synth.make_custom(T=40, d=64, E=32, k=6, f=32, fs=32, x_dtype="bf16", w_dtype="e4m3", seed=13)
    full = oracle.layer_forward(inp)
    sub = oracle.layer_forward_tokens(inp, [3, 17, 39])
    assert np.allclose(sub["y"], full["y"][[3, 17, 39]], rtol=1e-12, atol=1e-12)
    assert np.array_equal(sub["ids"], full["ids"][[3, 17, 39]])


def test_out_perm_rows_are_gate_weighted_expert_outputs():
    inp = moe_synth.make_custom(T=10, d=32, E=8, k=2, f=16, fs=16, x_dtype="f32", w_dtype="f32", seed=14)
    res = oracle.layer_forward(inp)
    x = oracle.x_values(inp)
    for r, p in enumerate(res["sorted_pair"]):
        t, j = divmod(int(p), 2)
        e = int(res["ids"][t, j])
        assert res["offsets"][e] <= r < res["offsets"][e + 1]
        W13, W2 = oracle.expert_weights(inp, e)
        assert np.allclose(res["out_perm"][r], res["w"][t, j] * _torch_swiglu(x[t:t + 1], W13, W2)[0],
                           rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- 8-bit activations
# (the restatement the library's opt-in MOE_FLAG_ACT_E4M3 mode is checked against)

def test_encode_e4m3_matches_torch_cast():
    rng = np.random.default_rng(21)
    v = np.clip(rng.standard_normal(4000) * 60, -448, 448).astype(np.float32).astype(np.float64)
    pos = oracle.moe_oracle._E4M3_POS
    mids = (pos[:-1] + pos[1:]) / 2                      # exact ties between neighbouring codes
    vals = np.concatenate([v, mids, -mids, pos, -pos])
    ref = torch.tensor(vals, dtype=torch.float32).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(oracle.encode_e4m3(vals), ref)


def test_act_scale_is_the_smallest_power_of_two():
    rng = np.random.default_rng(22)
    amaxes = np.concatenate([np.exp(rng.uniform(-60, 60, 400)), [448.0, 449.0, 224.0, 224.5, 3.5, 1.0, 1e-38]])
    for amax in amaxes:
        s = oracle.act_scale(float(amax))
        m, _ = math.frexp(s)
        assert m == 0.5                                   # a power of two
        assert amax <= 448.0 * s
        assert amax > 224.0 * s or s == 2.0 ** -126       # and no smaller one would do
    assert oracle.act_scale(448.0) == 1.0 and oracle.act_scale(448.5) == 2.0
    assert oracle.act_scale(0.0) == 1.0 and oracle.act_scale(float("nan")) == 1.0


def test_quantize_act_rows_error_bounds_and_idempotence():
    rng = np.random.default_rng(23)
    X = rng.standard_normal((6, 300)) * np.exp(rng.uniform(-6, 6, (6, 1)))
    Q = oracle.quantize_act_rows(X)
    for r in range(X.shape[0]):
        s = oracle.act_scale(float(np.abs(X[r]).max()))
        normal = np.abs(X[r]) >= 2.0 ** -6 * s
        err = np.abs(Q[r] - X[r])
        assert np.all(err[normal] <= 2.0 ** -4 * np.abs(X[r][normal]))   # half an ulp of 3 mantissa bits
        assert np.all(err[~normal] <= 2.0 ** -10 * s)                    # half the subnormal step
        assert np.abs(Q[r]).max() <= 448.0 * s
    assert np.array_equal(oracle.quantize_act_rows(Q), Q)


def test_round_bf16_matches_torch():
    rng = np.random.default_rng(24)
    v = (rng.standard_normal(3000) * np.exp(rng.uniform(-20, 20, 3000))).astype(np.float32)
    ref = torch.tensor(v).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(oracle.round_bf16(v.astype(np.float64)), ref)


def test_act_e4m3_ffn_is_near_but_not_equal():
    # the lossy mode stays within a few E4M3 roundings of the exact FFN
    rng = np.random.default_rng(25)
    X = rng.standard_normal((12, 64))
    W13 = rng.standard_normal((2 * 32, 64)) / 8
    W2 = rng.standard_normal((64, 32)) / 6
    exact = oracle.swiglu_ffn(X, W13, W2)
    lossy = oracle.swiglu_ffn(X, W13, W2, act="e4m3")
    rel = np.linalg.norm(lossy - exact) / np.linalg.norm(exact)
    assert 1e-3 < rel < 0.15
    # inputs already on the scaled E4M3 grid pass the first rounding unchanged
    Xq = oracle.quantize_act_rows(X)
    assert np.array_equal(oracle.quantize_act_rows(Xq), Xq)


# --------------------------------------------------------------------------
# The opt-in 8-bit-activation branch of swiglu_ffn, pinned as a whole: a
# hand-worked case (tests/golden/act_e4m3_example.json) in which the bf16
# rounding of H flips an E4M3 code, and an independent restatement with
# torch's own float8 / bfloat16 casts and a brute-force scale search.


def test_act_e4m3_hand_example():
    g = _load("act_e4m3_example.json")
    X = np.array(g["x"], dtype=np.float64)
    W13 = np.array(g["w13"], dtype=np.float64)
    W2 = np.array(g["w2"], dtype=np.float64)
    ex = g["expected"]
    assert np.array_equal(oracle.quantize_act_rows(X), np.array(ex["xq"]))
    out = oracle.swiglu_ffn(X, W13, W2, act="e4m3")
    assert np.allclose(out, np.array(ex["out"]), rtol=0, atol=1e-12)
    assert not np.allclose(out, np.array(ex["out_without_bf16_rounding_of_h"]), rtol=0, atol=1e-3)
    assert np.allclose(oracle.swiglu_ffn(X, W13, W2), np.array(ex["out_exact_activations"]), rtol=0, atol=1e-12)


def _torch_act_rows(V):
    """Per row: s = the smallest power of two with max|v| <= 448 s, found by
    walking every exponent; then torch's float8_e4m3fn cast of v / s."""
    out = torch.empty_like(V)
    for r in range(V.shape[0]):
        amax = float(V[r].abs().max())
        s = 1.0
        if amax > 0:
            for e in range(-126, 128):
                if amax <= 448.0 * 2.0 ** e:
                    s = 2.0 ** e
                    break
        out[r] = (V[r] / s).to(torch.float8_e4m3fn).to(torch.float64) * s
    return out


def test_act_e4m3_ffn_matches_torch_restatement():
    # dyadic weights keep every matmul exact in fp64, so the two sides must
    # agree bit for bit; rows of very different magnitudes exercise the scale
    rng = np.random.default_rng(26)
    d, f, n = 48, 24, 10
    X = rng.standard_normal((n, d)) * np.exp2(rng.integers(-6, 7, (n, 1)))
    W13 = rng.integers(-64, 65, (2 * f, d)) / 256.0
    W2 = rng.integers(-64, 65, (d, f)) / 256.0
    got = oracle.swiglu_ffn(X, W13, W2, act="e4m3")
    Xt, W13t, W2t = (torch.tensor(a, dtype=torch.float64) for a in (X, W13, W2))
    Xq = _torch_act_rows(Xt)
    G = torch.nn.functional.linear(Xq, W13t[:f])
    U = torch.nn.functional.linear(Xq, W13t[f:])
    H = (torch.nn.functional.silu(G) * U).to(torch.float32).to(torch.bfloat16).to(torch.float64)
    ref = torch.nn.functional.linear(_torch_act_rows(H), W2t).numpy()
    assert np.array_equal(got, ref)
    # and the rounding matters: exact activations give a different result
    assert not np.allclose(oracle.swiglu_ffn(X, W13, W2), ref, rtol=1e-3, atol=0)


# --------------------------------------------------------------------------
# The opt-in NVFP4-activation branch (W4A4): each rule restated by brute
# force, a hand-worked row (tests/golden/nvfp4_act_example.json) and the
# whole SwiGLU composition restated independently.


def test_nvfp4_act_hand_example():
    g = _load("nvfp4_act_example.json")
    row = np.array(g["row"], dtype=np.float64)
    ex = g["expected"]
    assert oracle.nvfp4_row_scale(float(np.abs(row).max())) == ex["g"]
    for b, s in enumerate(ex["block_scales"]):
        assert oracle.nvfp4_block_scale(float(np.abs(row[16 * b:16 * b + 16]).max()), ex["g"]) == s
    got = oracle.quantize_nvfp4_act_rows(row[None])[0]
    assert np.array_equal(got, np.array(ex["row"], dtype=np.float64))


def _e2m1_brute(x):
    """Nearest of the 15 E2M1 values by exhaustive search; a tie takes the
    value whose code (magnitude index) is even; beyond 6 saturates."""
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    a = min(abs(x), 6.0)
    best = min(range(8), key=lambda c: (abs(mags[c] - a), c % 2))
    return math.copysign(mags[best], x) if mags[best] else 0.0


def test_encode_e2m1_bruteforce():
    rng = np.random.default_rng(31)
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    v = np.concatenate([rng.uniform(-8, 8, 4000), mids, [-m for m in mids], [0.0, 6.0, 6.5, -100.0]])
    got = oracle.encode_e2m1(v)
    want = np.array([_e2m1_brute(float(x)) for x in v])
    assert np.array_equal(np.abs(got), np.abs(want)) and np.all((got == 0) | (np.sign(got) == np.sign(v)))


def test_nvfp4_scales_bruteforce():
    rng = np.random.default_rng(32)
    e4m3_pos = sorted({float(x) for x in oracle.E4M3_TABLE[1:0x7F]})
    for amax in np.concatenate([np.exp(rng.uniform(-40, 40, 300)), [2688.0, 2688.5, 1.0, 21.0]]):
        g = oracle.nvfp4_row_scale(float(amax))
        walk = next(2.0 ** e for e in range(-126, 128) if amax <= 2688.0 * 2.0 ** e)
        assert g == walk
        for frac in (1.0, 0.9, 0.31, 1e-3, 1e-6):
            b = float(amax) * frac
            s = oracle.nvfp4_block_scale(b, g)
            assert s == next(v for v in e4m3_pos if b <= 6.0 * g * v)   # scan of every positive code
    assert oracle.nvfp4_block_scale(0.0, 1.0) == 1.0 and oracle.nvfp4_row_scale(0.0) == 1.0


def _torch_nvfp4_rows(V):
    """Independent restatement: g by walking exponents, s by scanning the
    E4M3 codes through torch's float8_e4m3fn view, elements by exhaustive
    nearest-value search."""
    codes = torch.arange(1, 0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
    out = torch.empty_like(V)
    for r in range(V.shape[0]):
        amax = float(V[r].abs().max())
        g = next((2.0 ** e for e in range(-126, 128) if amax <= 2688.0 * 2.0 ** e), 1.0) if amax > 0 else 1.0
        for b in range(0, V.shape[1], 16):
            blk = V[r, b:b + 16]
            bm = float(blk.abs().max())
            s = float(codes[torch.nonzero(6.0 * g * codes >= bm)[0, 0]]) if bm > 0 else 1.0
            out[r, b:b + 16] = torch.tensor([_e2m1_brute(float(x) / (g * s)) for x in blk],
                                            dtype=torch.float64) * (g * s)
    return out


def test_act_nvfp4_ffn_matches_torch_restatement():
    # dyadic weights keep every matmul exact in fp64: bit-for-bit agreement
    rng = np.random.default_rng(33)
    d, f, n = 64, 32, 6
    X = rng.standard_normal((n, d)) * np.exp2(rng.integers(-5, 6, (n, 1)))
    W13 = rng.integers(-64, 65, (2 * f, d)) / 256.0
    W2 = rng.integers(-64, 65, (d, f)) / 256.0
    got = oracle.swiglu_ffn(X, W13, W2, act="nvfp4")
    Xt, W13t, W2t = (torch.tensor(a, dtype=torch.float64) for a in (X, W13, W2))
    Xq = _torch_nvfp4_rows(Xt)
    G = torch.nn.functional.linear(Xq, W13t[:f])
    U = torch.nn.functional.linear(Xq, W13t[f:])
    H = (torch.nn.functional.silu(G) * U).to(torch.float32).to(torch.bfloat16).to(torch.float64)
    ref = torch.nn.functional.linear(_torch_nvfp4_rows(H), W2t).numpy()
    assert np.array_equal(got, ref)
    assert not np.allclose(oracle.swiglu_ffn(X, W13, W2), ref, rtol=1e-2, atol=0)


def test_quantize_nvfp4_act_rows_error_bound():
    # every element within half the widest E2M1 step (1) of its block scale
    rng = np.random.default_rng(34)
    V = rng.standard_normal((5, 256)) * np.exp(rng.uniform(-5, 5, (5, 1)))
    Q = oracle.quantize_nvfp4_act_rows(V)
    for r in range(5):
        g = oracle.nvfp4_row_scale(float(np.abs(V[r]).max()))
        for b in range(0, 256, 16):
            s = oracle.nvfp4_block_scale(float(np.abs(V[r, b:b + 16]).max()), g)
            assert np.all(np.abs(Q[r, b:b + 16] - V[r, b:b + 16]) <= 1.0 * g * s)
            assert np.all(np.abs(Q[r, b:b + 16]) <= 6.0 * g * s)


def test_act_nvfp4_swiglu_hand_example():
    g = _load("nvfp4_swiglu_example.json")
    d = f = 16
    X = np.zeros((1, d))
    X[0, 0] = g["x_col0"]
    W13 = np.zeros((2 * f, d))
    W13[0, 0], W13[1, 0] = g["gate_col0"]
    W13[f, 0], W13[f + 1, 0] = g["up_col0"]
    out = oracle.swiglu_ffn(X, W13, np.eye(d), act="nvfp4")[0, :3]
    assert np.allclose(out, g["expected_out_first3"], rtol=0, atol=1e-12)
    assert not np.allclose(out, g["out_without_bf16_rounding_of_h_first3"], rtol=0, atol=1e-3)
