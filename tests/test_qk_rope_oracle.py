"""Pins of the QK-norm + RoPE oracle (oracle/qk_rope_oracle.py) against what
the mathematics and an independent library fix, and mutants that the pins
catch.  CPU only."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle.qk_rope_oracle as qr

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_hand_example():
    g = json.load(open(os.path.join(GOLDEN, "qk_rope_example.json")))
    x = np.array(g["x"])[None, None, :]
    cs = np.array(g["cos_sin"])[None]                     # one position
    qo, ko = qr.qk_norm_rope(x, x, g["gamma"], g["gamma"], cs, [0], eps=g["eps"])
    assert np.allclose(qo[0, 0], g["expected"], rtol=0, atol=1e-12)
    assert np.allclose(ko[0, 0], g["expected"], rtol=0, atol=1e-12)


def test_rms_norm_matches_torch():
    rng = np.random.default_rng(41)
    x = rng.standard_normal((7, 5, 128)) * np.exp(rng.uniform(-3, 3, (7, 5, 1)))
    gamma = rng.uniform(0.5, 1.5, 128)
    ref = torch.nn.functional.rms_norm(torch.tensor(x), (128,), torch.tensor(gamma), eps=1e-6).numpy()
    assert np.allclose(qr.rms_norm(x, gamma, 1e-6), ref, rtol=1e-12, atol=1e-12)


def test_rms_norm_closed_forms():
    # a constant row c: mean square c^2, so y = c / sqrt(c^2 + eps) * gamma
    g = np.linspace(0.5, 2.0, 64)
    for c in (3.0, -0.25, 1e-3):
        y = qr.rms_norm(np.full(64, c), g, 1e-6)
        assert np.allclose(y, c / math.sqrt(c * c + 1e-6) * g, rtol=1e-13)
    # scale invariance without eps
    x = np.random.default_rng(42).standard_normal(32)
    assert np.allclose(qr.rms_norm(7.5 * x, np.ones(32), 0.0), qr.rms_norm(x, np.ones(32), 0.0), rtol=1e-13)


def test_rope_identities():
    rng = np.random.default_rng(43)
    D, n_pos = 64, 50
    tab = qr.rope_table(n_pos, D)
    # the table: frequency 0 turns by one radian per position; angle addition
    assert np.allclose(tab[:, 0, 0], np.cos(np.arange(n_pos)), atol=1e-15)
    assert np.allclose(tab[:, 0, 1], np.sin(np.arange(n_pos)), atol=1e-15)
    m, n = 17, 23
    c = tab[m, :, 0] * tab[n, :, 0] - tab[m, :, 1] * tab[n, :, 1]
    s = tab[m, :, 1] * tab[n, :, 0] + tab[m, :, 0] * tab[n, :, 1]
    assert np.allclose(c, tab[m + n, :, 0], atol=1e-12) and np.allclose(s, tab[m + n, :, 1], atol=1e-12)
    y = rng.standard_normal((3, D))
    # position 0 is the identity; each (i, i + D/2) pair keeps its length
    assert np.allclose(qr.rope_rotate_half(y, tab[0, :, 0], tab[0, :, 1]), y, atol=1e-15)
    r = qr.rope_rotate_half(y, tab[m, :, 0], tab[m, :, 1])
    h = D // 2
    assert np.allclose(r[:, :h] ** 2 + r[:, h:] ** 2, y[:, :h] ** 2 + y[:, h:] ** 2, rtol=1e-12)
    # relative position: <R(m) u, R(n) v> = <R(m - n) u, v>
    u, v = rng.standard_normal(D), rng.standard_normal(D)
    lhs = np.dot(qr.rope_rotate_half(u, tab[m + n, :, 0], tab[m + n, :, 1]),
                 qr.rope_rotate_half(v, tab[n, :, 0], tab[n, :, 1]))
    rhs = np.dot(qr.rope_rotate_half(u, tab[m, :, 0], tab[m, :, 1]), v)
    assert abs(lhs - rhs) < 1e-10 * (1 + abs(rhs))


# --------------------------------------------------------------------------- mutants

def _rope_interleaved(y, cos, sin):
    y = np.asarray(y, dtype=np.float64)
    a, b = y[..., 0::2], y[..., 1::2]
    out = np.empty_like(y)
    out[..., 0::2] = a * cos - b * sin
    out[..., 1::2] = b * cos + a * sin
    return out


def _rope_sin_sign(y, cos, sin):
    h = y.shape[-1] // 2
    a, b = y[..., :h], y[..., h:]
    return np.concatenate([a * cos + b * sin, b * cos - a * sin], axis=-1)


def _norm_eps_outside(x, gamma, eps):
    x = np.asarray(x, dtype=np.float64)
    return x / (np.sqrt(np.mean(x * x, axis=-1, keepdims=True)) + eps) * gamma


def _norm_gamma_first(x, gamma, eps):
    z = np.asarray(x, dtype=np.float64) * gamma
    return z / np.sqrt(np.mean(z * z, axis=-1, keepdims=True) + eps)


MUTANTS = [
    ("rope_rotate_half", _rope_interleaved, test_hand_example),
    ("rope_rotate_half", _rope_interleaved, test_rope_identities),
    ("rope_rotate_half", _rope_sin_sign, test_hand_example),
    ("rms_norm", _norm_eps_outside, test_rms_norm_closed_forms),
    ("rms_norm", _norm_gamma_first, test_rms_norm_matches_torch),
]


@pytest.mark.parametrize("name,fn,pin", MUTANTS, ids=[f"{m[0]}:{m[1].__name__}:{m[2].__name__}" for m in MUTANTS])
def test_pin_catches_mutant(monkeypatch, name, fn, pin):
    monkeypatch.setattr(qr, name, fn)
    with pytest.raises(AssertionError):
        pin()
