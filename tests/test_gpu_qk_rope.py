"""GPU parity of the fused in-place QK-norm + RoPE step (moe_qk_norm_rope)
against the oracle, element by element.

Bound per element: |gpu - ref| <= 2^-8 |ref| + 1e-5 max|row of ref|.  The
kernel rounds its fp32 result to bf16 once (at most 2^-9 relative); its fp32
arithmetic adds about 1e-6 relative to the row's largest element (the
rotation's a cos - b sin can cancel), so the bound holds with a factor two
to spare."""
import numpy as np
import pytest
import torch

import moe_synth
from oracle import qk_rope_oracle as qr
from top_routed_expert_gb300 import abi
from top_routed_expert_gb300.layer import _to_dev

pytestmark = pytest.mark.gpu


def _bf16(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _run(inp, positions=None, eps=1e-6):
    dev = "cuda"
    q = _to_dev(inp.q, dev).clone()
    k = _to_dev(inp.k, dev).clone()
    pos = _to_dev(inp.positions if positions is None else positions, dev)
    cfg = abi.moe_qk_rope_config_t(inp.T, inp.n_q_heads, inp.n_kv_heads, inp.head_dim, inp.n_pos, eps)
    abi.moe_qk_norm_rope(cfg, q, k, _to_dev(inp.gamma_q, dev), _to_dev(inp.gamma_k, dev), _to_dev(inp.cos_sin, dev),
                         pos)
    st = abi.moe_get_device_status()
    return q.cpu().numpy().view(np.uint16), k.cpu().numpy().view(np.uint16), st


def _check(got_bits, ref):
    got = _bf16(got_bits)
    rowmax = np.max(np.abs(ref), axis=-1, keepdims=True)
    bound = 2.0 ** -8 * np.abs(ref) + 1e-5 * rowmax
    err = np.abs(got - ref)
    assert np.all(err <= bound), f"worst {np.max(err / np.maximum(bound, 1e-30)):.3f} of the bound"
    # and the rounding itself: nearly every element is the bf16 of the exact value
    exact = torch.tensor(ref).to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.mean(got_bits == exact) > 0.99


def _ref(inp):
    return qr.qk_norm_rope(_bf16(inp.q), _bf16(inp.k), inp.gamma_q, inp.gamma_k, inp.cos_sin, inp.positions)


def test_prefill_workload_every_element():
    inp = moe_synth.make_qk_inputs()            # T = 8192, 32 / 4 heads of 128, 4096 positions
    q, k, st = _run(inp)
    assert st == 0
    qo, ko = _ref(inp)
    _check(q, qo)
    _check(k, ko)


@pytest.mark.parametrize("T,hq,hkv,D", [(1, 1, 1, 128), (7, 3, 1, 64), (33, 8, 2, 256), (300, 32, 4, 128)])
def test_shapes(T, hq, hkv, D):
    inp = moe_synth.make_qk_inputs(T=T, n_q_heads=hq, n_kv_heads=hkv, head_dim=D, n_pos=600, chunk=37, prompt=600,
                                   seed=T + D)
    inp.positions[-1] = inp.n_pos - 1           # the last table row
    q, k, st = _run(inp)
    assert st == 0
    qo, ko = _ref(inp)
    _check(q, qo)
    _check(k, ko)


def test_out_of_range_position_is_reported_and_left_alone():
    inp = moe_synth.make_qk_inputs(T=40, n_q_heads=4, n_kv_heads=2, n_pos=64, chunk=8, prompt=64, seed=5)
    pos = inp.positions.copy()
    pos[3], pos[17] = 64, -1
    q, k, st = _run(inp, pos)
    assert st == 6                              # MOE_ERR_DEVICE_BOUNDS
    assert np.array_equal(q[[3, 17]], inp.q[[3, 17]]) and np.array_equal(k[[3, 17]], inp.k[[3, 17]])
    keep = np.setdiff1d(np.arange(40), [3, 17])
    qo, ko = qr.qk_norm_rope(_bf16(inp.q[keep]), _bf16(inp.k[keep]), inp.gamma_q, inp.gamma_k, inp.cos_sin, pos[keep])
    _check(q[keep], qo)
    _check(k[keep], ko)
    assert abi.moe_get_device_status() == 0


def test_deterministic_bitwise():
    inp = moe_synth.make_qk_inputs(T=1024, seed=3)
    a = _run(inp)
    b = _run(inp)
    assert a[2] == 0 and np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
