"""Seeded synthetic inputs for the MoE FFN layer (test and benchmark data only).

This package generates the inputs that both the CUDA path and the CPU oracle
consume: activations, router weights, per-expert bias (skewed workload only)
and the expert / shared-expert weights in their *stored* formats (FP8 E4M3
codes with per-output-channel fp32 scales, or NVFP4 packed e2m1 codes with
16-element E4M3 block scales and an fp32 global scale, or plain fp32).

It holds none of the layer's arithmetic: no logits, no routing, no FFN.  The
weight quantisers here play the role of the offline model-quantisation tool
the Sarvam blog names ("NVIDIA Model Optimizer", Blackwell section) and only
decide which codes are stored; the layer then consumes those codes as given.

Workloads (shapes from the Sarvam blog, "Scaling multilingual sovereign AI
with MoE": 128 experts, top-6 for the 30B shape, top-8 and FFN width 2048 for
the 100B shape; a shared expert in both):

  tiny          T=32,   d=128,  k=6, f=64,   all fp32
  decode        T=64,   d=4096, k=6, f=1024, FP8 weights, bf16 x
  prefill       T=8192, d=4096, k=6, f=1024, FP8 weights, bf16 x (32 x 256-token chunks)
  skew          T=4096, d=4096, k=6, f=1024, FP8, Zipf-biased router
  100b_decode   T=64,   d=4096, k=8, f=2048, NVFP4 weights, bf16 x
  100b_prefill  T=8192, d=4096, k=8, f=2048, NVFP4 weights, bf16 x

Value distributions: x ~ N(0,1) (rounded to bf16 where x is bf16); router,
expert and shared weights ~ N(0, 1/d_model) before quantisation.  Every
tensor draws from its own child of ``numpy.random.SeedSequence(seed)`` so a
single expert can be regenerated or inspected independently.
"""
from __future__ import annotations

import dataclasses
import math
import os
from concurrent.futures import ThreadPoolExecutor
from typing import Optional

import numpy as np
import torch

__all__ = ["CONFIGS", "MoEInputs", "make_inputs", "make_custom", "with_heavy_tails", "QKInputs", "make_qk_inputs",
           "bf16_bits_to_f32",
           "quantize_e4m3_rows", "quantize_nvfp4", "SKEW_C", "SKEW_DEAD"]


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int
    d: int
    E: int
    k: int
    f: int
    fs: int
    x_dtype: str      # "f32" | "bf16"
    w_dtype: str      # "f32" | "e4m3" | "nvfp4"
    skew: bool = False


CONFIGS = {
    "tiny": MoEConfig("tiny", 32, 128, 128, 6, 64, 64, "f32", "f32"),
    "decode": MoEConfig("decode", 64, 4096, 128, 6, 1024, 1024, "bf16", "e4m3"),
    "prefill": MoEConfig("prefill", 8192, 4096, 128, 6, 1024, 1024, "bf16", "e4m3"),
    "skew": MoEConfig("skew", 4096, 4096, 128, 6, 1024, 1024, "bf16", "e4m3", skew=True),
    "100b_decode": MoEConfig("100b_decode", 64, 4096, 128, 8, 2048, 2048, "bf16", "nvfp4"),
    "100b_prefill": MoEConfig("100b_prefill", 8192, 4096, 128, 8, 2048, 2048, "bf16", "nvfp4"),
}

# Zipf-skew router bias: bias_e = -SKEW_C * 1.2 * ln(rank_e), rank_e a seeded
# permutation of 1..E, and the SKEW_DEAD lowest-ranked experts get -30 so that
# some groups are certainly empty.  SKEW_C was chosen by
# tests/golden/calibrate_skew.py (which routes with the oracle) so that the
# hottest expert receives about 8x the mean load at T=4096, seed 0.
SKEW_C = 0.3087
SKEW_DEAD = 4
SKEW_S = 1.2


@dataclasses.dataclass
class MoEInputs:
    cfg: MoEConfig
    x: np.ndarray                 # [T,d] float32 (f32 configs) or uint16 bf16 bits
    w_router: np.ndarray          # [E,d] float32
    bias: Optional[np.ndarray]    # [E] float32 or None
    # routed experts, stored formats (see module docstring)
    w13: np.ndarray               # f32 [E,2f,d] | e4m3 u8 [E,2f,d] | nvfp4 u8 [E,2f,d/2]
    w13_scale: Optional[np.ndarray]   # e4m3: f32 [E,2f]; nvfp4: u8 e4m3 codes [E,2f,d/16]
    w13_gscale: Optional[np.ndarray]  # nvfp4: f32 [E]
    w2: np.ndarray                # f32 [E,d,f] | u8 [E,d,f] | u8 [E,d,f/2]
    w2_scale: Optional[np.ndarray]
    w2_gscale: Optional[np.ndarray]
    # shared expert, same formats with a leading dim of 1
    s13: np.ndarray
    s13_scale: Optional[np.ndarray]
    s13_gscale: Optional[np.ndarray]
    s2: np.ndarray
    s2_scale: Optional[np.ndarray]
    s2_gscale: Optional[np.ndarray]

    @property
    def x_f32(self) -> np.ndarray:
        """x as float32 values (exact for bf16 storage)."""
        if self.cfg.x_dtype == "bf16":
            return bf16_bits_to_f32(self.x)
        return self.x


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def _f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def quantize_e4m3_rows(w: np.ndarray):
    """Per-output-channel FP8 E4M3: s_n = amax(row n)/448, q = RNE(w/s_n).

    Returns (codes uint8 [..., rows, K], scales float32 [..., rows]).  A zero
    row gets scale 1.  Rounding is torch's float8_e4m3fn cast (round to
    nearest even); inputs are clamped to +-448 first so nothing saturates to
    NaN.
    """
    w = np.asarray(w, dtype=np.float32)
    amax = np.max(np.abs(w), axis=-1)
    s = (amax / np.float32(448.0)).astype(np.float32)
    s[s == 0] = np.float32(1.0)
    v = np.clip(w / s[..., None], -448.0, 448.0).astype(np.float32)
    q = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return q, s


# e2m1 magnitude grid, code 0..7 (sign in bit 3)
_E2M1_MID = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], dtype=np.float32)


def _e2m1_encode(v: np.ndarray) -> np.ndarray:
    """Nearest e2m1 code of v (ties to the even code), saturating at 6."""
    mag = np.abs(v)
    code = np.searchsorted(_E2M1_MID, mag, side="left").astype(np.int32)
    lo = np.minimum(code, 6)
    tie = (code < 7) & (mag == _E2M1_MID[lo]) & ((code & 1) == 1)
    code = code + tie.astype(np.int32)
    code = np.minimum(code, 7)
    sign = ((v < 0) & (code > 0)).astype(np.int32) << 3
    return (code | sign).astype(np.uint8)


def quantize_nvfp4(w: np.ndarray):
    """NVFP4 for one matrix [rows, K] (K a multiple of 32).

    g = amax(matrix)/(6*448) (fp32 global scale); per 16-element block along
    K, s_b = e4m3(amax(block)/(6 g)) (a block whose scale code is zero gets
    code 0x38 = 1.0); q = nearest e2m1 of w/(s_b g).  Two codes per byte along
    K: element 2i in the low nibble, element 2i+1 in the high nibble.
    Returns (packed u8 [rows, K/2], block-scale codes u8 [rows, K/16], g f32).
    """
    w = np.asarray(w, dtype=np.float32)
    rows, K = w.shape
    amax = float(np.max(np.abs(w)))
    g = np.float32(amax / (6.0 * 448.0)) if amax > 0 else np.float32(1.0)
    blk = w.reshape(rows, K // 16, 16)
    bamax = np.max(np.abs(blk), axis=-1)
    sreal = np.clip(bamax / (np.float32(6.0) * g), 0, 448.0).astype(np.float32)
    scode = torch.from_numpy(sreal).to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()
    scode[scode == 0] = 0x38
    sval = torch.from_numpy(scode).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    v = blk / (sval[..., None] * g)
    codes = _e2m1_encode(v.astype(np.float32)).reshape(rows, K)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return packed, scode, g


def _normal(ss: np.random.SeedSequence, shape, std: float) -> np.ndarray:
    rng = np.random.default_rng(ss)
    a = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return a


def _make_matrix(ss, rows, K, std, w_dtype):
    w = _normal(ss, (rows, K), std)
    if w_dtype == "f32":
        return w, None, None
    if w_dtype == "e4m3":
        q, s = quantize_e4m3_rows(w)
        return q, s, None
    if w_dtype == "nvfp4":
        return quantize_nvfp4(w)
    raise ValueError(w_dtype)


def _stack(parts):
    out = []
    for i in range(3):
        if parts[0][i] is None:
            out.append(None)
        else:
            out.append(np.stack([p[i] for p in parts]))
    return out


def make_inputs(name_or_cfg, seed: int = 0, threads: Optional[int] = None,
                router_only: bool = False, skew_c: Optional[float] = None) -> MoEInputs:
    """Build the seeded synthetic inputs of one workload.

    router_only skips the expert weights (they are left as None); skew_c
    overrides SKEW_C (used only by the calibration script)."""
    cfg = CONFIGS[name_or_cfg] if isinstance(name_or_cfg, str) else name_or_cfg
    T, d, E, k, f, fs = cfg.T, cfg.d, cfg.E, cfg.k, cfg.f, cfg.fs
    root = np.random.SeedSequence(seed)
    ss_x, ss_wr, ss_skew, ss_shared, *ss_exp = root.spawn(4 + E)
    std = 1.0 / math.sqrt(d)

    xf = _normal(ss_x, (T, d), 1.0)
    x = _f32_to_bf16_bits(xf) if cfg.x_dtype == "bf16" else xf
    w_router = _normal(ss_wr, (E, d), std)

    bias = None
    if cfg.skew:
        rank = np.random.default_rng(ss_skew).permutation(E) + 1
        c = SKEW_C if skew_c is None else skew_c
        bias = (-c * SKEW_S * np.log(rank.astype(np.float64))).astype(np.float32)
        bias[rank > E - SKEW_DEAD] = np.float32(-30.0)

    if router_only:
        return MoEInputs(cfg, x, w_router, bias, *([None] * 12))

    def expert(i):
        c13, c2 = ss_exp[i].spawn(2)
        return (_make_matrix(c13, 2 * f, d, std, cfg.w_dtype),
                _make_matrix(c2, d, f, std, cfg.w_dtype))

    nthreads = threads or min(32, max(1, len(os.sched_getaffinity(0))))
    with ThreadPoolExecutor(nthreads) as ex:
        parts = list(ex.map(expert, range(E)))
    w13, w13_s, w13_g = _stack([p[0] for p in parts])
    w2, w2_s, w2_g = _stack([p[1] for p in parts])

    sh13, sh2 = ss_shared.spawn(2)
    s13, s13_s, s13_g = _stack([_make_matrix(sh13, 2 * fs, d, std, cfg.w_dtype)])
    s2, s2_s, s2_g = _stack([_make_matrix(sh2, d, fs, std, cfg.w_dtype)])

    return MoEInputs(cfg, x, w_router, bias, w13, w13_s, w13_g, w2, w2_s, w2_g,
                     s13, s13_s, s13_g, s2, s2_s, s2_g)


def make_custom(T, d, E, k, f, fs, x_dtype="f32", w_dtype="f32", seed=0, skew=False) -> MoEInputs:
    """Inputs for an ad-hoc shape (small edge-case tests)."""
    return make_inputs(MoEConfig(f"custom_T{T}_d{d}_E{E}_k{k}_f{f}", T, d, E, k, f, fs,
                                 x_dtype, w_dtype, skew), seed)


def with_heavy_tails(inp: MoEInputs, per_row: int = 3, magnitude: float = 1000.0, seed: int = 0) -> MoEInputs:
    """A copy of `inp` whose activations carry a heavy tail: in every token
    row, `per_row` seeded positions are set to +-magnitude (random signs,
    rounded to the activation dtype).  Activation outliers of this kind stretch
    a per-row scale far above most of the row's elements."""
    rng = np.random.default_rng(seed)
    xf = np.array(inp.x_f32, dtype=np.float32, copy=True)
    T, d = xf.shape
    for t in range(T):
        cols = rng.choice(d, size=per_row, replace=False)
        xf[t, cols] = np.float32(magnitude) * rng.choice(np.array([-1.0, 1.0], dtype=np.float32), size=per_row)
    x = _f32_to_bf16_bits(xf) if inp.cfg.x_dtype == "bf16" else xf
    return dataclasses.replace(inp, x=x)


# ---------------------------------------------------------------------------
# Inputs of the fused QK-norm + RoPE step (attention block of the same
# model: d_model 4096 = 32 query heads of width 128, grouped-query attention
# with 4 key heads).  A prefill batch of 32 requests x 256-token chunks, each
# request's chunk at a seeded offset inside a 3584-token prompt (the pages'
# input sequence length); the frequency table covers 4096 positions.


@dataclasses.dataclass
class QKInputs:
    T: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    q: np.ndarray           # [T][Hq][D] uint16 bf16 bits
    k: np.ndarray           # [T][Hkv][D] uint16 bf16 bits
    gamma_q: np.ndarray     # [D] float32
    gamma_k: np.ndarray     # [D] float32
    cos_sin: np.ndarray     # [n_pos][D/2][2] float32
    positions: np.ndarray   # [T] int32

    @property
    def n_pos(self) -> int:
        return self.cos_sin.shape[0]


def make_qk_inputs(T=8192, n_q_heads=32, n_kv_heads=4, head_dim=128, n_pos=4096, chunk=256, prompt=3584,
                   theta=10000.0, seed=0) -> QKInputs:
    """q, k ~ N(0,1) with a seeded log-normal scale per (token, head) row
    (so the normalisation has something to do), gammas ~ U(0.5, 1.5), the
    (cos, sin) table of pos * theta^(-2i/D) rounded to float32, positions of
    consecutive chunks at seeded offsets."""
    ss = np.random.SeedSequence(seed).spawn(6)
    rq, rk, rg, rp = (np.random.default_rng(x) for x in ss[:4])
    qf = rq.standard_normal((T, n_q_heads, head_dim), dtype=np.float32)
    qf *= np.exp(rq.standard_normal((T, n_q_heads, 1))).astype(np.float32)
    kf = rk.standard_normal((T, n_kv_heads, head_dim), dtype=np.float32)
    kf *= np.exp(rk.standard_normal((T, n_kv_heads, 1))).astype(np.float32)
    gq = rg.uniform(0.5, 1.5, head_dim).astype(np.float32)
    gk = rg.uniform(0.5, 1.5, head_dim).astype(np.float32)
    i = np.arange(head_dim // 2, dtype=np.float64)
    ang = np.arange(n_pos, dtype=np.float64)[:, None] * theta ** (-2.0 * i / head_dim)[None, :]
    cs = np.stack([np.cos(ang), np.sin(ang)], axis=-1).astype(np.float32)
    n_req = (T + chunk - 1) // chunk
    offs = rp.integers(0, max(1, min(prompt, n_pos) - chunk + 1), n_req)
    t = np.arange(T)
    pos = (offs[t // chunk] + t % chunk).astype(np.int32)
    return QKInputs(T, n_q_heads, n_kv_heads, head_dim, _f32_to_bf16_bits(qf), _f32_to_bf16_bits(kf), gq, gk, cs, pos)
