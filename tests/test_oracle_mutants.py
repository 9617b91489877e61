"""Plant plausible mistakes in the oracle and check that a pin catches each.

Every mutant replaces one oracle function (in both the package namespace and
the implementation module) for the duration of one test, then runs the pin
that should fail.  The mutants are CPU-only and never touch the CUDA path.
"""
import math

import numpy as np
import pytest

import oracle
import oracle.moe_oracle as om
import tests.test_oracle as pins


def _patch(monkeypatch, name, fn):
    monkeypatch.setattr(om, name, fn)
    monkeypatch.setattr(oracle, name, fn)


def _tiebreak_high(L, k):
    T, E = L.shape
    idx = np.broadcast_to(np.arange(E), (T, E))
    return np.lexsort((-idx, -L), axis=1)[:, :k].astype(np.int32)


def _gates_no_renorm(L, ids):
    p = np.exp(L - L.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    return np.take_along_axis(p, ids.astype(np.int64), 1)


def _silu_wrong_sign(z):
    return z / (1.0 + np.exp(z))


def _swiglu_swapped(X, W13, W2, act=None):
    f = W2.shape[1]
    return (om.silu(X @ W13[f:].T) * (X @ W13[:f].T)) @ W2.T


def _swiglu_w2_transposed(X, W13, W2, act=None):
    f = W2.shape[1]
    return (om.silu(X @ W13[:f].T) * (X @ W13[f:].T)) @ W2


def _permute_by_token(ids, E):
    c, o, sp, r = _orig_permute(ids, E)
    # mistake: order within an expert by slot j first instead of by pair index
    k = ids.shape[1]
    out = sp.copy()
    for e in range(E):
        seg = out[o[e]:o[e + 1]]
        out[o[e]:o[e + 1]] = seg[np.lexsort((seg // k, seg % k))]
    r2 = np.empty_like(out)
    r2[out] = np.arange(out.size, dtype=np.int32)
    return c, o, out, r2


_orig_permute = om.permute
_orig_table = om.E4M3_TABLE.copy()


def _logits_ignore_bias(x, w_router, bias):
    return np.asarray(x, np.float64) @ np.asarray(w_router, np.float64).T


def _e2m1_nibbles_swapped(packed):
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.float64)
    out[..., 0::2] = om.E2M1_TABLE[p >> 4]
    out[..., 1::2] = om.E2M1_TABLE[p & 0xF]
    return out


def _swiglu_no_silu(X, W13, W2, act=None):
    f = W2.shape[1]
    return ((X @ W13[:f].T) * (X @ W13[f:].T)) @ W2.T


def _encode_truncating(v):
    v = np.asarray(v, dtype=np.float64)
    pos = om._E4M3_POS
    i = np.clip(np.searchsorted(pos, np.abs(v), side="right") - 1, 0, 126)
    return np.sign(v) * pos[i]


def _act_scale_doubled(amax):
    return 2.0 * _orig_act_scale(amax)


_orig_act_scale = om.act_scale


def _swiglu_e4m3_h_not_bf16(X, W13, W2, act=None):
    # mistake: the 8-bit branch quantises H straight from fp64
    f = W2.shape[1]
    if act == "e4m3":
        X = om.quantize_act_rows(X)
    H = om.silu(X @ W13[:f].T) * (X @ W13[f:].T)
    if act == "e4m3":
        H = om.quantize_act_rows(H)
    return H @ W2.T


def _swiglu_e4m3_h_unquantised(X, W13, W2, act=None):
    # mistake: the 8-bit branch quantises X but leaves H at bf16
    f = W2.shape[1]
    if act == "e4m3":
        X = om.quantize_act_rows(X)
    H = om.silu(X @ W13[:f].T) * (X @ W13[f:].T)
    if act == "e4m3":
        H = om.round_bf16(H)
    return H @ W2.T


def _swiglu_e4m3_x_unquantised(X, W13, W2, act=None):
    # mistake: the 8-bit branch quantises H only
    f = W2.shape[1]
    H = om.silu(X @ W13[:f].T) * (X @ W13[f:].T)
    if act == "e4m3":
        H = om.quantize_act_rows(om.round_bf16(H))
    return H @ W2.T


def _e2m1_ties_away(v):
    # mistake: ties rounded away from zero instead of to the even code
    v = np.asarray(v, dtype=np.float64)
    pos = om._E2M1_POS
    a = np.minimum(np.abs(v), 6.0)
    i = np.clip(np.searchsorted(pos, a, side="right") - 1, 0, 6)
    up = a - pos[i] >= pos[i + 1] - a
    return np.sign(v) * pos[np.where(up, i + 1, i)]


def _block_scale_nearest(bamax, g):
    # mistake: block scale rounded to the nearest E4M3 value (can saturate elements)
    t = np.asarray(bamax, dtype=np.float64) / (6.0 * np.asarray(g, dtype=np.float64))
    i = np.argmin(np.abs(om._E4M3_POS[1:][None, :] - np.reshape(t, (-1, 1))), axis=1) + 1
    return np.where(np.asarray(bamax) > 0, om._E4M3_POS[i].reshape(np.shape(t)), 1.0)


def _row_scale_exact(amax):
    # mistake: the row scale is amax / 2688 itself, not a power of two
    return amax / 2688.0 if amax > 0 and math.isfinite(amax) else 1.0


def _swiglu_nvfp4_h_not_bf16(X, W13, W2, act=None):
    # mistake: the NVFP4 branch quantises H straight from fp64
    f = W2.shape[1]
    if act == "nvfp4":
        X = om.quantize_nvfp4_act_rows(X)
    H = om.silu(X @ W13[:f].T) * (X @ W13[f:].T)
    if act == "nvfp4":
        H = om.quantize_nvfp4_act_rows(H)
    return H @ W2.T


MUTANTS = [
    ("topk_ids", _tiebreak_high, pins.test_topk_bruteforce_with_exact_ties, (8, 3)),
    ("gates", _gates_no_renorm, pins.test_gates_special_cases, ()),
    ("gates", _gates_no_renorm, pins.test_hand_example, ()),
    ("silu", _silu_wrong_sign, pins.test_silu_special_values, ()),
    ("swiglu_ffn", _swiglu_swapped, pins.test_swiglu_matches_torch, ()),
    ("swiglu_ffn", _swiglu_w2_transposed, pins.test_swiglu_matches_torch, ()),
    ("swiglu_ffn", _swiglu_no_silu, pins.test_hand_example, ()),
    ("permute", _permute_by_token, pins.test_permute_bruteforce_and_invariants, (7, 8, 3)),
    ("router_logits", _logits_ignore_bias, pins.test_router_logits_bias_and_linearity, ()),
    ("decode_e2m1_packed", _e2m1_nibbles_swapped, pins.test_e2m1_packing_nibble_order, ()),
    ("encode_e4m3", _encode_truncating, pins.test_encode_e4m3_matches_torch_cast, ()),
    ("act_scale", _act_scale_doubled, pins.test_act_scale_is_the_smallest_power_of_two, ()),
    ("swiglu_ffn", _swiglu_e4m3_h_not_bf16, pins.test_act_e4m3_hand_example, ()),
    ("swiglu_ffn", _swiglu_e4m3_h_not_bf16, pins.test_act_e4m3_ffn_matches_torch_restatement, ()),
    ("swiglu_ffn", _swiglu_e4m3_h_unquantised, pins.test_act_e4m3_hand_example, ()),
    ("swiglu_ffn", _swiglu_e4m3_h_unquantised, pins.test_act_e4m3_ffn_matches_torch_restatement, ()),
    ("swiglu_ffn", _swiglu_e4m3_x_unquantised, pins.test_act_e4m3_hand_example, ()),
    ("swiglu_ffn", _swiglu_e4m3_x_unquantised, pins.test_act_e4m3_ffn_matches_torch_restatement, ()),
    ("encode_e2m1", _e2m1_ties_away, pins.test_encode_e2m1_bruteforce, ()),
    ("encode_e2m1", _e2m1_ties_away, pins.test_nvfp4_act_hand_example, ()),
    ("nvfp4_block_scale", _block_scale_nearest, pins.test_nvfp4_scales_bruteforce, ()),
    ("nvfp4_block_scale", _block_scale_nearest, pins.test_act_nvfp4_ffn_matches_torch_restatement, ()),
    ("nvfp4_row_scale", _row_scale_exact, pins.test_nvfp4_act_hand_example, ()),
    ("nvfp4_row_scale", _row_scale_exact, pins.test_act_nvfp4_ffn_matches_torch_restatement, ()),
    ("swiglu_ffn", _swiglu_nvfp4_h_not_bf16, pins.test_act_nvfp4_swiglu_hand_example, ()),
]


@pytest.mark.parametrize("name,fn,pin,args", MUTANTS, ids=[f"{m[0]}:{m[1].__name__}:{m[2].__name__}" for m in MUTANTS])
def test_pin_catches_mutant(monkeypatch, name, fn, pin, args):
    _patch(monkeypatch, name, fn)
    with pytest.raises(AssertionError):
        pin(*args)


def test_pin_catches_e4m3_exponent_bias(monkeypatch):
    bad = np.array([om._e4m3_value(c) * 0.5 for c in range(256)])   # bias 8 instead of 7
    monkeypatch.setattr(om, "E4M3_TABLE", bad)
    monkeypatch.setattr(oracle, "E4M3_TABLE", bad)
    with pytest.raises(AssertionError):
        pins.test_e4m3_table_matches_torch_cast()


def test_pin_catches_dropped_shared_expert(monkeypatch):
    def no_shared(inp):
        W13, W2 = _orig_shared(inp)
        return W13, W2 * 0.0
    _orig_shared = om.shared_weights
    _patch(monkeypatch, "shared_weights", no_shared)
    with pytest.raises(AssertionError):
        pins.test_hand_example()


def test_unmutated_pins_pass():
    for _, _, pin, args in MUTANTS:
        pin(*args)
    assert math.isfinite(float(om.E4M3_TABLE[0x7E]))
