"""GPU parity of the whole layer and of each ABI call against the CPU oracle.

Every workload is compared on every token: routing bit for bit (outside the
reported near ties) and the layer output element by element (the oracle
dequantises one expert at a time, so the full-size workloads take tens of
seconds on the host cores)."""
import numpy as np
import pytest
import torch

import moe_synth
import oracle
from top_routed_expert_gb300 import abi
from top_routed_expert_gb300.layer import MoELayer

from .gpu_util import LOSSY_MAX_ABS_RMS, check_output, check_routing, device_x, oracle_y, run_layer, workload

pytestmark = pytest.mark.gpu

PATHS = [pytest.param(0, id="default"), pytest.param(abi.MOE_FLAG_SIMT_FFN, id="simt")]


@pytest.mark.parametrize("flags", PATHS)
@pytest.mark.parametrize("name", ["tiny", "decode", "100b_decode"])
def test_full_workload_elementwise(name, flags):
    inp = workload(name)
    _, _, y, ids, w, offs = run_layer(inp, flags)
    check_routing(inp, ids, w, offs)
    check_output(inp, y, ids)


@pytest.mark.parametrize("flags", PATHS)
@pytest.mark.parametrize("name", ["prefill", "skew", "100b_prefill"])
def test_full_workload_every_token(name, flags):
    # all T tokens element by element: every expert's ragged last token tile
    # and every weight tile of the full-size batches
    inp = workload(name)
    _, _, y, ids, w, offs = run_layer(inp, flags)
    check_routing(inp, ids, w, offs)
    check_output(inp, y, ids)
    assert np.all(np.isfinite(y))


@pytest.mark.parametrize("flags", PATHS)
@pytest.mark.parametrize("w_dtype", ["e4m3", "nvfp4"])
def test_heavy_tailed_activations(w_dtype, flags):
    # decode shape with a few activations per token at about 1000 sigma: the
    # row scale follows the outliers, so most elements sit far below it (the
    # two-term E4M3 split's inexact range below 2^-6 of the scale, the f16
    # row scaling's lowest bits), and H inherits the heavy tail
    f = 1024 if w_dtype == "e4m3" else 2048
    inp = moe_synth.with_heavy_tails(
        moe_synth.make_custom(T=64, d=4096, E=128, k=6 if w_dtype == "e4m3" else 8, f=f, fs=f, x_dtype="bf16",
                              w_dtype=w_dtype, seed=77), per_row=3, magnitude=1000.0, seed=78)
    _, _, y, ids, w, offs = run_layer(inp, flags)
    check_routing(inp, ids, w, offs)
    check_output(inp, y, ids)


@pytest.mark.parametrize("flags", PATHS)
@pytest.mark.parametrize("w_dtype", ["f32", "e4m3", "nvfp4"])
@pytest.mark.parametrize("x_dtype", ["f32", "bf16"])
def test_ragged_shapes(w_dtype, x_dtype, flags):
    # several row tiles per expert, a ragged last tile, f != f_s, d not a power of two
    inp = moe_synth.make_custom(T=301, d=384, E=16, k=4, f=192, fs=128, x_dtype=x_dtype, w_dtype=w_dtype, seed=21)
    _, _, y, ids, w, offs = run_layer(inp, flags)
    check_routing(inp, ids, w, offs)
    check_output(inp, y, ids)


@pytest.mark.parametrize("T,E,k", [(1, 8, 1), (5, 8, 8), (40, 1, 1), (17, 256, 16), (3, 128, 6)])
def test_edge_shapes(T, E, k):
    inp = moe_synth.make_custom(T=T, d=256, E=E, k=k, f=64, fs=64, x_dtype="bf16", w_dtype="e4m3", seed=T + E)
    _, _, y, ids, w, offs = run_layer(inp)
    check_routing(inp, ids, w, offs)
    check_output(inp, y, ids)
    if k == 1:
        assert np.all(w == 1.0)


@pytest.mark.parametrize("w_dtype", ["e4m3", "nvfp4"])
def test_largest_hidden_size(w_dtype):
    # d_model = 16384, the largest the ABI accepts: the router's widest
    # slices and the row quantisers' loop path (rows longer than 4096)
    inp = moe_synth.make_custom(T=40, d=16384, E=8, k=2, f=128, fs=128, x_dtype="bf16", w_dtype=w_dtype, seed=16)
    _, _, y, ids, w, offs = run_layer(inp)
    check_routing(inp, ids, w, offs)
    check_output(inp, y, ids)


def test_skew_has_empty_and_hot_experts():
    inp = workload("skew")
    _, _, _, ids, _, offs = run_layer(inp)
    counts = np.diff(offs)
    assert (counts == 0).sum() >= 4
    assert counts.max() / counts.mean() > 7.5


def test_bf16_output():
    # y rounded to bf16 once more: the stated tolerance plus half a bf16 ulp
    # (2^-9 relative) of each output element
    inp = workload("decode")
    _, _, y, ids, _, _ = run_layer(inp, y_dtype=abi.MOE_BF16)
    check_output(inp, y, ids, ulp_rel=2.0 ** -9)


def test_zero_tokens():
    inp = moe_synth.make_custom(T=4, d=128, E=8, k=2, f=64, fs=64, x_dtype="bf16", w_dtype="e4m3")
    layer = MoELayer(inp)
    x = device_x(inp)[:0]
    y = layer.forward(x)
    assert y.shape == (0, 128)
    assert abi.moe_get_device_status() == 0


@pytest.mark.parametrize("name", ["decode", "100b_decode", "prefill"])
def test_deterministic_bitwise(name):
    # three passes over the same input give identical bits (no atomics, a
    # fixed summation order everywhere; a race in a pipeline hand-off would
    # show up here even when it stays inside the parity tolerance)
    inp = workload(name)
    layer = MoELayer(inp)
    x = device_x(inp)
    y1 = layer.forward(x).clone()
    for _ in range(2):
        assert torch.equal(layer.forward(x), y1)
    assert abi.moe_get_device_status() == 0


@pytest.mark.parametrize("flags", [0, abi.MOE_FLAG_BF16_EXPERT_OUT])
def test_stepwise_calls_match_layer_forward(flags):
    inp = moe_synth.make_custom(T=96, d=256, E=32, k=6, f=128, fs=128, x_dtype="bf16", w_dtype="e4m3", seed=5)
    layer = MoELayer(inp, flags=flags)
    x = device_x(inp)
    y_full = layer.forward(x)
    cfg = layer.config()
    T, k, E, d = inp.cfg.T, inp.cfg.k, inp.cfg.E, inp.cfg.d
    dev = "cuda"
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    offs = torch.empty(E + 1, dtype=torch.int32, device=dev)
    sp = torch.empty(T * k, dtype=torch.int32, device=dev)
    row_of = torch.empty(T * k, dtype=torch.int32, device=dev)
    edt = torch.bfloat16 if flags else torch.float32
    out_perm = torch.empty((T * k, d), dtype=edt, device=dev)
    shared = torch.empty((T, d), dtype=edt, device=dev)
    y = torch.empty((T, d), dtype=torch.float32, device=dev)
    ws = layer.workspace()
    abi.moe_route(cfg, x, layer.w_router, layer.bias, ids, w, ws)
    abi.moe_permute(cfg, ids, offs, sp, row_of, ws)
    abi.moe_expert_ffn(cfg, x, w, offs, sp, layer.weights, out_perm, shared, ws)
    abi.moe_combine(cfg, out_perm, row_of, shared, y)
    assert abi.moe_get_device_status() == 0
    assert torch.equal(y, y_full)
    # permutation: bit-exact against the oracle's on the same ids
    c_ref, o_ref, sp_ref, r_ref = oracle.permute(ids.cpu().numpy(), E)
    assert np.array_equal(offs.cpu().numpy(), o_ref)
    assert np.array_equal(sp.cpu().numpy(), sp_ref)
    assert np.array_equal(row_of.cpu().numpy(), r_ref)
    # out_perm rows and the shared output, element by element
    ref = oracle.layer_forward(inp)
    ids_np = ids.cpu().numpy()
    assert np.array_equal(ids_np, ref["ids"])
    for name, got, want in (("out_perm", out_perm, ref["out_perm"]), ("shared", shared, ref["shared"])):
        g = got.float().cpu().numpy().astype(np.float64)
        rel = np.linalg.norm(g - want) / np.linalg.norm(want)
        assert rel < 5e-3, (name, rel)


@pytest.mark.parametrize("P_mult", [1, 7])
def test_permute_bit_exact_large(P_mult):
    # many chunks of the counting sort; random ids with empty experts
    E, k = 128, 6
    T = 2048 * P_mult + 5
    rng = np.random.default_rng(P_mult)
    ids = np.stack([rng.choice(E - 3, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    cfg = abi.make_config(T, 128, E, k, 64, 64)
    dev = "cuda"
    ids_d = torch.from_numpy(ids).to(dev)
    offs = torch.empty(E + 1, dtype=torch.int32, device=dev)
    sp = torch.empty(T * k, dtype=torch.int32, device=dev)
    row_of = torch.empty(T * k, dtype=torch.int32, device=dev)
    ws = torch.empty(abi.moe_workspace_bytes(cfg), dtype=torch.uint8, device=dev)
    abi.moe_permute(cfg, ids_d, offs, sp, row_of, ws)
    assert abi.moe_get_device_status() == 0
    c_ref, o_ref, sp_ref, r_ref = oracle.permute(ids, E)
    assert np.array_equal(offs.cpu().numpy(), o_ref)
    assert np.array_equal(sp.cpu().numpy(), sp_ref)
    assert np.array_equal(row_of.cpu().numpy(), r_ref)


def test_out_of_range_ids_reported_not_faulted():
    E, k, T = 16, 2, 100
    ids = np.tile(np.array([[0, 1]], dtype=np.int32), (T, 1))
    ids[7, 1] = 99          # corrupt
    ids[50, 0] = -3
    cfg = abi.make_config(T, 128, E, k, 64, 64)
    dev = "cuda"
    offs = torch.empty(E + 1, dtype=torch.int32, device=dev)
    sp = torch.zeros(T * k, dtype=torch.int32, device=dev)
    row_of = torch.zeros(T * k, dtype=torch.int32, device=dev)
    ws = torch.empty(abi.moe_workspace_bytes(cfg), dtype=torch.uint8, device=dev)
    abi.moe_permute(cfg, torch.from_numpy(ids).to(dev), offs, sp, row_of, ws)
    assert abi.moe_get_device_status() == 6     # MOE_ERR_DEVICE_BOUNDS
    assert offs.cpu().numpy()[-1] == T * k - 2
    r = row_of.cpu().numpy()
    assert r[7 * k + 1] == -1 and r[50 * k + 0] == -1   # skipped slots are marked for the combine
    assert sorted(np.delete(r, [7 * k + 1, 50 * k])) == list(range(T * k - 2))
    assert abi.moe_get_device_status() == 0     # cleared


def test_router_alone_with_bias():
    inp = moe_synth.make_custom(T=77, d=512, E=64, k=5, f=64, fs=64, x_dtype="bf16", w_dtype="e4m3", seed=9)
    inp.bias = np.linspace(-2, 2, 64).astype(np.float32)
    layer = MoELayer(inp)
    cfg = layer.config()
    ids = torch.empty((77, 5), dtype=torch.int32, device="cuda")
    w = torch.empty((77, 5), dtype=torch.float32, device="cuda")
    abi.moe_route(cfg, device_x(inp), layer.w_router, layer.bias, ids, w, layer.workspace())
    assert abi.moe_get_device_status() == 0
    ids_np, w_np = ids.cpu().numpy(), w.cpu().numpy()
    _, o = check_routing(inp, ids_np, w_np, oracle.permute(ids_np, 64)[1])


def _route(inp, x=None):
    layer = MoELayer(inp)
    T, k = inp.cfg.T, inp.cfg.k
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    abi.moe_route(layer.config(), device_x(inp) if x is None else x, layer.w_router, layer.bias, ids, w,
                  layer.workspace())
    return ids.cpu().numpy(), w.cpu().numpy(), abi.moe_get_device_status()


# T = 77 runs the CUDA-core router, T = 1100 the tensor-core router
@pytest.mark.parametrize("T", [77, 1100])
def test_exact_ties_take_the_lower_expert(T):
    # identical router rows give bitwise-equal logits in both routers (same
    # operands, same accumulation order): the lower expert index must come
    # first whenever the higher one is picked
    E, k = 16, 4
    inp = moe_synth.make_custom(T=T, d=256, E=E, k=k, f=64, fs=64, x_dtype="bf16", w_dtype="e4m3", seed=T)
    twins = {5: 2, 9: 2, 12: 7}
    for hi, lo in twins.items():
        inp.w_router[hi] = inp.w_router[lo]
    ids, w, st = _route(inp)
    assert st == 0
    hits = 0
    for t in range(T):
        row = list(ids[t])
        for hi, lo in twins.items():
            if hi in row:
                assert lo in row and row.index(lo) < row.index(hi), (t, row)
                assert w[t, row.index(lo)] == w[t, row.index(hi)]
                hits += 1
    assert hits > 0


@pytest.mark.parametrize("T", [77, 1100])
def test_nonfinite_input_is_reported(T):
    # a token with an infinite input has no finite logit: the status word
    # says so, and every other token routes exactly as in a clean run
    inp = moe_synth.make_custom(T=T, d=256, E=32, k=4, f=64, fs=64, x_dtype="bf16", w_dtype="e4m3", seed=3)
    ids0, w0, st0 = _route(inp)
    assert st0 == 0
    x = device_x(inp)
    x[3, 0] = 0x7F80    # bf16 +inf bit pattern
    ids1, w1, st1 = _route(inp, x)
    assert st1 == 8     # MOE_ERR_DEVICE_NONFINITE
    keep = np.arange(T) != 3
    assert np.array_equal(ids0[keep], ids1[keep]) and np.array_equal(w0[keep], w1[keep])
    assert abi.moe_get_device_status() == 0     # cleared


# Opt-in 8-bit activations (MOE_FLAG_ACT_E4M3): parity against the oracle's
# restatement of that rounding; the exact-activation oracle is a few percent
# away, which is what the mode trades for half the MMA work.
@pytest.mark.parametrize("name", ["decode", "prefill"])
def test_act_e4m3_matches_its_oracle(name):
    inp = workload(name)
    _, _, y, ids, w, offs = run_layer(inp, abi.MOE_FLAG_ACT_E4M3)
    check_routing(inp, ids, w, offs)
    tokens = np.arange(inp.cfg.T)
    check_output(inp, y, ids, tokens, act="e4m3")
    exact = oracle_y(inp, tokens, ids[tokens])
    rel = np.linalg.norm(y[tokens] - exact) / np.linalg.norm(exact)
    assert 5e-3 < rel < 0.15, rel


@pytest.mark.parametrize("shape", [dict(T=64, d=256, E=16, k=2, f=128, fs=256),
                                   dict(T=301, d=384, E=16, k=4, f=256, fs=384)], ids=["T64", "T301"])
def test_act_e4m3_tiles(shape):
    inp = moe_synth.make_custom(x_dtype="bf16", w_dtype="e4m3", seed=shape["T"] + 1, **shape)
    _, _, y, ids, w, offs = run_layer(inp, abi.MOE_FLAG_ACT_E4M3)
    check_routing(inp, ids, w, offs)
    check_output(inp, y, ids, act="e4m3")


# Shapes whose average rows per expert select each tensor-core token tile
# (TN = 8, 16, 32, 64, 128) with ragged last tiles, f != f_s, and a d that is
# not a power of two.
TC_SHAPES = [
    dict(T=20, d=384, E=32, k=2, f=256, fs=128),     # ~1 row / expert   -> TN 8
    dict(T=64, d=256, E=16, k=2, f=128, fs=256),     # 8 rows / expert   -> TN 16
    dict(T=100, d=384, E=16, k=2, f=256, fs=128),    # 12.5              -> TN 32
    dict(T=160, d=256, E=16, k=4, f=128, fs=128),    # 40                -> TN 64
    dict(T=301, d=384, E=16, k=4, f=256, fs=384),    # 75                -> TN 128
    dict(T=500, d=384, E=8, k=4, f=256, fs=128),     # 250: TN 128 (FP8), 256 (NVFP4 f16 rebuild)
]


@pytest.mark.parametrize("w_dtype", ["e4m3", "nvfp4"])
@pytest.mark.parametrize("shape", TC_SHAPES, ids=[f"T{s['T']}_E{s['E']}" for s in TC_SHAPES])
def test_tensor_core_path_tiles(shape, w_dtype):
    inp = moe_synth.make_custom(x_dtype="bf16", w_dtype=w_dtype, seed=shape["T"], **shape)
    _, _, y, ids, w, offs = run_layer(inp)
    check_routing(inp, ids, w, offs)
    check_output(inp, y, ids)


# Shapes that put the FP8 GEMMs on CTA pairs (M = 256 over two SMs): routed
# groups above 48 rows on average and d, f, f_s multiples of 256; ragged last
# token tiles in every group, several 256-row weight tiles per group.
PAIR_SHAPES = [
    dict(T=200, d=512, E=16, k=4, f=256, fs=512),    # 50 rows / expert: TN 64 (gate/up), 128 (down)
    dict(T=777, d=768, E=8, k=2, f=512, fs=256),     # 194 rows / expert, 3 down tiles of 256 rows
    dict(T=203, d=256, E=2, k=1, f=256, fs=256),     # 101 rows / expert, k = 1, one weight tile per group
]


@pytest.mark.parametrize("act", [None, "e4m3"])
@pytest.mark.parametrize("shape", PAIR_SHAPES, ids=[f"T{s['T']}_E{s['E']}" for s in PAIR_SHAPES])
def test_cta_pair_tiles(shape, act):
    inp = moe_synth.make_custom(x_dtype="bf16", w_dtype="e4m3", seed=shape["T"] + 3, **shape)
    flags = abi.MOE_FLAG_ACT_E4M3 if act else 0
    _, _, y, ids, w, offs = run_layer(inp, flags)
    check_routing(inp, ids, w, offs)
    check_output(inp, y, ids, act=act)


def test_cta_pair_bf16_expert_outputs():
    # the pair down projection's bf16 store branch: one more bf16 rounding of
    # each expert output (about 2^-9 relative), hence the wider element bound
    shape = PAIR_SHAPES[0]
    inp = moe_synth.make_custom(x_dtype="bf16", w_dtype="e4m3", seed=shape["T"] + 5, **shape)
    _, _, y, ids, w, offs = run_layer(inp, abi.MOE_FLAG_BF16_EXPERT_OUT)
    check_routing(inp, ids, w, offs)
    check_output(inp, y, ids, max_abs_rms=LOSSY_MAX_ABS_RMS)


@pytest.mark.parametrize("name", ["decode", "100b_decode"])
def test_tensor_core_matches_simt_closely(name):
    # both paths against each other: the exact activation encodings (two E4M3
    # terms, or scaled f16) keep the tensor-core result within bf16-rounding
    # distance (H is rounded to bf16 once) of the fp32 CUDA-core result
    inp = workload(name)
    _, _, y_tc, ids_tc, _, _ = run_layer(inp, 0)
    _, _, y_s, ids_s, _, _ = run_layer(inp, abi.MOE_FLAG_SIMT_FFN)
    assert np.array_equal(ids_tc, ids_s)
    rel = np.linalg.norm(y_tc - y_s) / np.linalg.norm(y_s)
    assert rel < 3e-3, rel


@pytest.mark.parametrize("T,E,k", [(1100, 96, 5), (1024, 128, 8), (2049, 128, 6)])
def test_tensor_core_router_ragged(T, E, k):
    # >= 1024 bf16 tokens and E <= 128 select the tensor-core router; a ragged
    # last 64-token tile, an E that leaves padded expert rows, and a bias
    inp = moe_synth.make_custom(T=T, d=512, E=E, k=k, f=128, fs=128, x_dtype="bf16", w_dtype="e4m3", seed=T)
    inp.bias = np.random.default_rng(T).standard_normal(E).astype(np.float32) * 0.5
    layer = MoELayer(inp)
    cfg = layer.config()
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    abi.moe_route(cfg, device_x(inp), layer.w_router, layer.bias, ids, w, layer.workspace())
    assert abi.moe_get_device_status() == 0
    ids_np, w_np = ids.cpu().numpy(), w.cpu().numpy()
    check_routing(inp, ids_np, w_np, oracle.permute(ids_np, E)[1])


def test_tensor_core_router_matches_cuda_core_router():
    inp = workload("prefill")
    out = []
    for flags in (0, abi.MOE_FLAG_SIMT_ROUTER):
        layer = MoELayer(inp, flags=flags)
        cfg = layer.config()
        T, k = inp.cfg.T, inp.cfg.k
        ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
        w = torch.empty((T, k), dtype=torch.float32, device="cuda")
        abi.moe_route(cfg, device_x(inp), layer.w_router, layer.bias, ids, w, layer.workspace())
        assert abi.moe_get_device_status() == 0
        out.append((ids.cpu().numpy(), w.cpu().numpy()))
    (i0, w0), (i1, w1) = out
    L = oracle.router_logits(oracle.x_values(inp), inp.w_router, None)
    sel, order = oracle.near_ties(L, inp.cfg.k)
    clean = ~sel & ~order
    assert np.array_equal(i0[clean], i1[clean])
    assert np.max(np.abs(w0[clean] - w1[clean])) < 1e-5
    for ids_np, w_np in out:
        check_routing(inp, ids_np, w_np, oracle.permute(ids_np, inp.cfg.E)[1])


def test_graph_capture_replays_the_layer():
    # the whole layer records into one CUDA graph; replays on new inputs match
    # the direct calls bit for bit
    inp = workload("decode")
    layer = MoELayer(inp)
    x = device_x(inp)
    graph, y = layer.capture(x)
    ref1 = layer.forward(x).clone()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(y, ref1)
    x2 = torch.roll(x, 1, dims=0)
    x.copy_(x2)
    ref2 = layer.forward(x).clone()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(y, ref2)
    assert abi.moe_get_device_status() == 0


# NVFP4 weights on the block-scaled FP4 MMA (the default for widths that are
# multiples of 256, decode-sized batches): activations as four NVFP4 terms.
# Shapes whose average rows per expert select each token tile (TN = 4, 8,
# 16; MMA N = 4 TN) with ragged last tiles, f != f_s, several weight tiles per
# group.
NVF4_SHAPES = [
    dict(T=12, d=256, E=32, k=4, f=256, fs=512),     # 1.5 rows / expert  -> TN 4
    dict(T=20, d=512, E=32, k=4, f=256, fs=512),     # 2.5                -> TN 8
    dict(T=100, d=512, E=16, k=2, f=512, fs=256),    # 12.5               -> TN 16
    dict(T=128, d=512, E=16, k=2, f=256, fs=768),    # 16 (most groups ragged) -> TN 16
]


@pytest.mark.parametrize("shape", NVF4_SHAPES, ids=[f"T{s['T']}_E{s['E']}" for s in NVF4_SHAPES])
def test_nvfp4_block_scaled_tiles(shape):
    inp = moe_synth.make_custom(x_dtype="bf16", w_dtype="nvfp4", seed=shape["T"] + 7, **shape)
    _, _, y, ids, w, offs = run_layer(inp)
    check_routing(inp, ids, w, offs)
    check_output(inp, y, ids)


@pytest.mark.parametrize("name", ["100b_decode", "100b_prefill"])
def test_nvfp4_f16_path_every_token(name):
    # the f16-rebuild path, kept for widths the block-scaled path does not take
    inp = workload(name)
    _, _, y, ids, w, offs = run_layer(inp, abi.MOE_FLAG_NVFP4_F16)
    check_routing(inp, ids, w, offs)
    check_output(inp, y, ids)


def test_nvfp4_paths_agree_closely():
    # four activation terms against the exact f16 rebuild: both within
    # bf16-rounding distance of each other (H is rounded to bf16 in both)
    inp = workload("100b_decode")
    _, _, y4, ids4, _, _ = run_layer(inp, 0)
    _, _, yh, idsh, _, _ = run_layer(inp, abi.MOE_FLAG_NVFP4_F16)
    assert np.array_equal(ids4, idsh)
    rel = np.linalg.norm(y4 - yh) / np.linalg.norm(yh)
    assert rel < 3e-3, rel


# Opt-in NVFP4 activations (MOE_FLAG_ACT_NVFP4, W4A4): parity against the
# oracle's restatement of that rounding; the exact-activation oracle is about
# a tenth away.
@pytest.mark.parametrize("name", ["100b_decode", "100b_prefill"])
def test_act_nvfp4_matches_its_oracle(name):
    inp = workload(name)
    _, _, y, ids, w, offs = run_layer(inp, abi.MOE_FLAG_ACT_NVFP4)
    check_routing(inp, ids, w, offs)
    tokens = np.arange(inp.cfg.T)
    check_output(inp, y, ids, tokens, act="nvfp4")
    exact = oracle_y(inp, tokens, ids[tokens])
    rel = np.linalg.norm(y[tokens] - exact) / np.linalg.norm(exact)
    assert 2e-2 < rel < 0.3, rel


ACT_NVF4_SHAPES = [
    dict(T=64, d=256, E=16, k=2, f=256, fs=512),     # 8 rows / expert -> TN 16
    dict(T=301, d=512, E=16, k=4, f=256, fs=256),    # 75             -> TN 128
]


@pytest.mark.parametrize("shape", ACT_NVF4_SHAPES, ids=["T64", "T301"])
def test_act_nvfp4_tiles(shape):
    inp = moe_synth.make_custom(x_dtype="bf16", w_dtype="nvfp4", seed=shape["T"] + 3, **shape)
    _, _, y, ids, w, offs = run_layer(inp, abi.MOE_FLAG_ACT_NVFP4)
    check_routing(inp, ids, w, offs)
    check_output(inp, y, ids, act="nvfp4")


# The shared expert beside the routing (a second stream inside
# moe_layer_forward) changes no arithmetic: the same bits as the layer with
# everything on one stream, on each FFN path.
@pytest.mark.parametrize("name,flags", [("decode", 0), ("prefill", 0), ("100b_decode", 0),
                                        ("100b_prefill", 0), ("decode", abi.MOE_FLAG_ACT_E4M3),
                                        ("100b_decode", abi.MOE_FLAG_ACT_NVFP4)])
def test_shared_expert_overlap_is_bitwise_neutral(name, flags):
    inp = workload(name)
    x = device_x(inp)
    y_split = MoELayer(inp, flags=flags).forward(x).clone()
    y_one = MoELayer(inp, flags=flags | abi.MOE_FLAG_NO_OVERLAP).forward(x)
    assert abi.moe_get_device_status() == 0
    assert torch.equal(y_split, y_one)


def test_overlapped_layer_captures_and_replays():
    # the fork and join record into the graph; replays track new inputs
    inp = workload("100b_decode")
    layer = MoELayer(inp)
    x = device_x(inp)
    graph, y = layer.capture(x)
    x.copy_(torch.roll(x, 3, dims=0))
    graph.replay()
    torch.cuda.synchronize()
    ref = MoELayer(inp, flags=abi.MOE_FLAG_NO_OVERLAP).forward(x)
    assert torch.equal(y, ref)
    assert abi.moe_get_device_status() == 0
