"""Shared helpers of the GPU parity tests: run the CUDA layer through the C
ABI and compare its outputs with the CPU oracle on the same seeded inputs."""
import functools

import numpy as np
import torch

import moe_synth
import oracle
from top_routed_expert_gb300 import abi
from top_routed_expert_gb300.layer import MoELayer, _to_dev

# Tolerances of the layer output (relative L2 error, max abs error relative
# to the rms of the reference output).
REL_L2 = 5e-3
MAX_ABS_RMS = 2e-2
# The opt-in lossy activation modes are compared with the oracle's
# restatement of their rounding.  Both sides take the same rounding
# decisions except where the GPU's fp32 H and the oracle's fp64 H straddle a
# bf16 rounding boundary (about 2^-15 of the elements); such an element can
# then move by one E4M3 / E2M1 step, or move its NVFP4 block's scale and so
# all 16 elements of the block.  The relative-L2 bound stays; a single output
# element may carry up to twice the default bound.
LOSSY_MAX_ABS_RMS = 4e-2
# Gate weights: fp32 logits carry ~1e-6 absolute error over d = 4096 terms;
# a gate moves by about the logit error times the gate.
GATE_ATOL = 2e-5


@functools.lru_cache(maxsize=4)
def workload(name, seed=0):
    return moe_synth.make_inputs(name, seed=seed)


def device_x(inp):
    return _to_dev(inp.x, "cuda")


def run_layer(inp, flags=0, y_dtype=abi.MOE_F32):
    layer = MoELayer(inp, flags=flags, y_dtype=y_dtype)
    x = device_x(inp)
    y, ids, w, offs = layer.forward(x, routing=True)
    st = abi.moe_get_device_status()
    assert st == 0, abi.STATUS.get(st, st)
    return layer, x, y.float().cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy(), offs.cpu().numpy()


def check_routing(inp, ids_gpu, w_gpu, offs_gpu):
    """ids bit-exact except near-tie tokens; gates within GATE_ATOL;
    offsets bit-exact against the oracle's permutation of the same choice."""
    k, E = inp.cfg.k, inp.cfg.E
    x = oracle.x_values(inp)
    L, ids_ref, _ = oracle.route(x, inp.w_router, inp.bias, k)
    sel, order = oracle.near_ties(L, k)
    clean = ~sel & ~order
    assert np.array_equal(ids_gpu[clean], ids_ref[clean]), "ids differ on tokens without near ties"
    ot = order & ~sel
    assert np.array_equal(np.sort(ids_gpu[ot], 1), np.sort(ids_ref[ot], 1)), "selected sets differ"
    # near-tie tokens may pick either side of the tie; every pick must still be
    # a valid top-k within the tie window
    for t in np.nonzero(sel)[0]:
        s = np.sort(L[t])[::-1]
        assert np.all(L[t, ids_gpu[t]] >= s[k - 1] - 1e-4)
    # gates of the GPU's own selection
    w_ref = oracle.gates(L, ids_gpu)
    assert np.max(np.abs(w_gpu - w_ref)) <= GATE_ATOL
    assert np.max(np.abs(w_gpu.sum(1) - 1.0)) <= k * 2.0 ** -22
    # counts / offsets: the oracle's own ids, with near-tie tokens taking the GPU's pick
    ids_mix = ids_ref.copy()
    ids_mix[sel] = ids_gpu[sel]
    _, offs_ref, _, _ = oracle.permute(ids_mix, E)
    assert np.array_equal(offs_gpu, offs_ref)
    return int(sel.sum()), int(order.sum())


# (workload, rel_l2, max_abs/rms) of every output check, reported at the end
# of the session by tests/conftest.py
PARITY_LOG = []


# oracle outputs already computed in this session, keyed by the input object,
# the tokens, the routing they were computed for and the activation mode (the
# full-size workloads take tens of seconds each on the host cores).  Each
# entry keeps its input object alive, so no later object can reuse its id.
_ORACLE_Y = {}


def oracle_y(inp, tokens, ids, act=None):
    key = (id(inp), np.asarray(tokens).tobytes(), np.asarray(ids).tobytes(), act)
    hit = _ORACLE_Y.get(key)
    if hit is None or hit[0] is not inp:
        if len(_ORACLE_Y) >= 8:
            _ORACLE_Y.clear()
        hit = (inp, oracle.layer_forward_tokens(inp, tokens, ids_override=ids, act=act)["y"])
        _ORACLE_Y[key] = hit
    return hit[1]


def check_output(inp, y_gpu, ids_gpu, tokens=None, max_abs_rms=MAX_ABS_RMS, ulp_rel=0.0, act=None):
    """rel-L2 <= REL_L2 and, element by element, |err| <= max_abs_rms * rms(y_ref)
    + ulp_rel * |y_ref| (ulp_rel = 0 except for a bf16 output, where one
    rounding of the output itself is allowed on top).  act = "e4m3" compares
    against the oracle's restatement of the 8-bit-activation mode.  tokens =
    None compares every token."""
    if tokens is None:
        tokens = np.arange(inp.cfg.T)
    ref = oracle_y(inp, tokens, ids_gpu[tokens], act)
    got = y_gpu[tokens].astype(np.float64)
    err = got - ref
    rel = np.linalg.norm(err) / np.linalg.norm(ref)
    rms = np.sqrt(np.mean(ref ** 2))
    mx = np.max(np.abs(err)) / rms
    PARITY_LOG.append((inp.cfg.name + (f"+act_{act}" if act else ""), float(rel), float(mx)))
    if act is not None:
        max_abs_rms = max(max_abs_rms, LOSSY_MAX_ABS_RMS)
    bound = max_abs_rms * rms + ulp_rel * np.abs(ref)
    assert rel <= REL_L2 and np.all(np.abs(err) <= bound), f"rel_l2={rel:.3e} max_abs/rms={mx:.3e}"
    return rel, mx
