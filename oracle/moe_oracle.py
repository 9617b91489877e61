"""CPU fp64 oracle of the Sarvam-style MoE FFN layer forward pass.

TEST INFRASTRUCTURE.  This module is the slow, obviously-correct reference the
CUDA path is checked against.  Only the tests, the smoke check of the package
entry point and the benchmark's CPU-baseline leg may import it; the library's
own code never does.  It shares no code with the CUDA path: it decodes the
stored weight codes itself, from the formats' bit-level definitions.

What the layer computes (sources, by page and section):

* Sarvam blog = NVIDIA technical blog "How NVIDIA extreme hardware-software
  co-design delivered a large inference boost for Sarvam AI's sovereign
  models".  Section "Scaling multilingual sovereign AI with MoE": 128 experts,
  top-6 routing (30B) / top-8 with MoE FFN hidden size 2048 (100B), plus a
  shared expert.  Table 1 rows "Router logits and TopK", "Routed expert
  compute", "Shared expert compute": the layer is router logits, a top-k
  selection, the routed experts and the shared expert, summed per token.
* Sarvam summary = peacm.com news/791474, section 2.1 (expert weights stored
  in FP8, one byte per parameter; a shared expert for general features plus
  routed experts) and section 3.1 (the fused router kernel writes expert
  indices and scores).
* InferX page (ijyty.com news/984491), section 2.4: probabilities are a
  softmax over the expert logits followed by a top-k; section 3.3: the router
  emits int32 indices and fp32 weights per token.

Readings where the pages are silent (the plainest reading in each case):
  softmax scoring; gates renormalised over the selected k; ties broken by the
  lowest expert index; one shared expert with weight 1; SwiGLU experts
  (silu(gate) * up, then down) with gate rows first in W13; an optional
  per-expert router bias added to the logits before selection.

Every function computes in float64.  Expert weights are dequantised one
expert at a time so host memory stays bounded.

Parity pins live in tests/test_oracle.py; none of the functions here is
"parity unpinned".
"""
from __future__ import annotations

import math
from typing import Dict, Iterable, Optional

import numpy as np

# --------------------------------------------------------------------------
# Number formats (bit-level definitions)
# --------------------------------------------------------------------------


def _e4m3_value(code: int) -> float:
    """FP8 E4M3 ("fn" variant): 1 sign, 4 exponent (bias 7), 3 mantissa bits;
    exponent 0 is subnormal (m/8 * 2^-6); code S.1111.111 is NaN; no inf."""
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def _e2m1_value(code: int) -> float:
    """FP4 E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; exponent 0 is
    subnormal (m * 0.5).  No inf / NaN."""
    s = -1.0 if code & 0x8 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        return s * m * 0.5
    return s * (1.0 + m / 2.0) * 2.0 ** (e - 1)


E4M3_TABLE = np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)
E2M1_TABLE = np.array([_e2m1_value(c) for c in range(16)], dtype=np.float64)


def decode_bf16(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns -> float64 (bf16 is the top half of an IEEE fp32)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def decode_e4m3(codes: np.ndarray) -> np.ndarray:
    return E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


def decode_e2m1_packed(packed: np.ndarray) -> np.ndarray:
    """[..., K/2] bytes -> [..., K] values; element 2i is the low nibble."""
    p = np.asarray(packed, dtype=np.uint8)
    lo = E2M1_TABLE[p & 0xF]
    hi = E2M1_TABLE[p >> 4]
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.float64)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def dequant(w_dtype: str, codes, scale=None, gscale=None) -> np.ndarray:
    """One stored weight matrix [rows, K] -> float64.

    f32   : the values themselves.
    e4m3  : value = e4m3(code) * scale[row]        (per output channel).
    nvfp4 : value = e2m1(code) * e4m3(bscale[row, k//16]) * gscale.
    """
    if w_dtype == "f32":
        return np.asarray(codes, dtype=np.float64)
    if w_dtype == "e4m3":
        return decode_e4m3(codes) * np.asarray(scale, dtype=np.float64)[:, None]
    if w_dtype == "nvfp4":
        v = decode_e2m1_packed(codes)
        bs = decode_e4m3(scale)                       # [rows, K/16]
        return v * np.repeat(bs, 16, axis=1) * float(gscale)
    raise ValueError(w_dtype)


# --------------------------------------------------------------------------
# Router: logits, softmax, top-k, renormalised gates
# --------------------------------------------------------------------------


def router_logits(x: np.ndarray, w_router: np.ndarray, bias: Optional[np.ndarray]) -> np.ndarray:
    """L[t,e] = sum_i x[t,i] * W_r[e,i] (+ b[e]).  [T,E] float64."""
    L = np.asarray(x, np.float64) @ np.asarray(w_router, np.float64).T
    if bias is not None:
        L = L + np.asarray(bias, np.float64)[None, :]
    return L


def topk_ids(L: np.ndarray, k: int) -> np.ndarray:
    """The first k experts in the order (descending logit, ascending index).

    np.lexsort sorts by the last key first: primary key -L, secondary e.
    """
    T, E = L.shape
    idx = np.broadcast_to(np.arange(E), (T, E))
    order = np.lexsort((idx, -L), axis=1)
    return order[:, :k].astype(np.int32)


def gates(L: np.ndarray, ids: np.ndarray) -> np.ndarray:
    """Softmax over all E restricted to the selected ids and renormalised to
    sum to one; the common factor cancels, leaving a softmax over the k
    selected logits (shifted by the largest for range)."""
    sel = np.take_along_axis(L, ids.astype(np.int64), axis=1)
    z = np.exp(sel - sel[:, :1])
    return z / z.sum(axis=1, keepdims=True)


def route(x, w_router, bias, k):
    L = router_logits(x, w_router, bias)
    ids = topk_ids(L, k)
    return L, ids, gates(L, ids)


def near_ties(L: np.ndarray, k: int, eps: float = 1e-4):
    """Tokens whose routing the fp64 logits do not pin against fp32 rounding.

    sel[t]   : the k-th and (k+1)-th largest logits differ by < eps, so the
               selected *set* may legitimately differ.
    order[t] : two adjacent logits inside the top k differ by < eps, so the
               *order* of ids (and of the gates) may differ.
    """
    s = -np.sort(-L, axis=1)
    E = L.shape[1]
    sel = np.zeros(L.shape[0], dtype=bool)
    if k < E:
        sel = (s[:, k - 1] - s[:, k]) < eps
    order = np.zeros(L.shape[0], dtype=bool)
    if k > 1:
        order = np.any((s[:, : k - 1] - s[:, 1:k]) < eps, axis=1)
    return sel, order


# --------------------------------------------------------------------------
# Permutation into per-expert groups
# --------------------------------------------------------------------------


def permute(ids: np.ndarray, E: int):
    """Group the T*k (token, slot) pairs by expert.

    pair p = t*k + j.  counts[e] = #pairs routed to e; offsets = exclusive
    prefix sum (offsets[E] = T*k); sorted_pair lists the pairs ordered by
    (expert, p) -- within an expert this is ascending token because a token
    picks an expert at most once; row_of is the inverse permutation.
    """
    flat = np.asarray(ids, dtype=np.int64).reshape(-1)
    counts = np.bincount(flat, minlength=E).astype(np.int32)
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    sorted_pair = np.argsort(flat, kind="stable").astype(np.int32)
    row_of = np.empty_like(sorted_pair)
    row_of[sorted_pair] = np.arange(sorted_pair.size, dtype=np.int32)
    return counts, offsets, sorted_pair, row_of


# --------------------------------------------------------------------------
# Optional 8-bit activations.  The default layer uses the activations as
# they are.  The opt-in lossy mode of the library (one E4M3 term per
# activation row) is checked against this restatement of its rounding:
#   row scale  s = the smallest power of two (>= 2^-126) with max|v| <= 448 s
#              (1 for a row without a non-zero finite maximum);
#   value      s * E4M3(v / s), E4M3 = nearest value, ties to the even code;
#   H          rounded to fp32, then to bf16 (nearest even) before that.
# The pages fix only the weight formats; this is the 8-bit-activation
# reading of their FP8 compute.
# --------------------------------------------------------------------------

# finite non-negative E4M3 values, code 0 .. 126 (ascending with the code)
_E4M3_POS = np.array([_e4m3_value(c) for c in range(0x7F)], dtype=np.float64)


def encode_e4m3(v: np.ndarray) -> np.ndarray:
    """Nearest E4M3 value of each element, ties to the even code, saturating
    at +-448 (returns the values, not the codes)."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    i = np.clip(np.searchsorted(_E4M3_POS, a, side="right") - 1, 0, 125)   # value(i) <= a < value(i+1)
    lo, hi = _E4M3_POS[i], _E4M3_POS[i + 1]
    up = (a - lo > hi - a) | ((a - lo == hi - a) & ((i & 1) == 1))
    code = np.where(up, i + 1, i)
    code = np.where(a >= _E4M3_POS[126], 126, code)
    return np.sign(v) * _E4M3_POS[code]


def act_scale(amax: float) -> float:
    """The smallest power of two s >= 2^-126 with amax <= 448 s."""
    if not (amax > 0.0) or not math.isfinite(amax):
        return 1.0
    k = max(math.ceil(math.log2(amax / 448.0)), -126)
    while k > -126 and amax <= 448.0 * 2.0 ** (k - 1):   # exact comparisons settle the log's rounding
        k -= 1
    while amax > 448.0 * 2.0 ** k:
        k += 1
    return 2.0 ** k


def quantize_act_rows(V: np.ndarray) -> np.ndarray:
    """Each row v -> s * E4M3(v / s) with its own scale s = act_scale(max|v|)."""
    V = np.asarray(V, dtype=np.float64)
    out = np.empty_like(V)
    for r in range(V.shape[0]):
        s = act_scale(float(np.max(np.abs(V[r]))) if V.shape[1] else 0.0)
        out[r] = encode_e4m3(V[r] / s) * s
    return out


# --------------------------------------------------------------------------
# Optional NVFP4 activations (the W4A4 reading of the Blackwell section's
# NVFP4 compute: activations in the same element format as the weights).
# The opt-in W4A4 mode of the library is checked against this restatement:
#   row scale    g = the smallest power of two (>= 2^-126) with
#                max|v| <= 6 * 448 * g  (1 for a row without a non-zero
#                finite maximum);
#   block scale  per 16 consecutive elements, s = the smallest positive E4M3
#                value with max|v_block| <= 6 * g * s  (1 for an all-zero
#                block), so no element saturates;
#   value        g * s * E2M1(v / (g s)), E2M1 = nearest value of
#                {0, 0.5, 1, 1.5, 2, 3, 4, 6}, ties to the even code;
#   H            rounded to fp32, then to bf16, before that.
# --------------------------------------------------------------------------

# non-negative E2M1 values by code 0 .. 7 (ascending with the code)
_E2M1_POS = np.array([_e2m1_value(c) for c in range(8)], dtype=np.float64)


def encode_e2m1(v: np.ndarray) -> np.ndarray:
    """Nearest E2M1 value of each element, ties to the even code, saturating
    at +-6 (returns the values, not the codes)."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    i = np.clip(np.searchsorted(_E2M1_POS, a, side="right") - 1, 0, 6)   # value(i) <= a < value(i+1)
    lo, hi = _E2M1_POS[i], _E2M1_POS[i + 1]
    up = (a - lo > hi - a) | ((a - lo == hi - a) & ((i & 1) == 1))
    code = np.where(up, i + 1, i)
    code = np.where(a >= 6.0, 7, code)
    return np.sign(v) * _E2M1_POS[code]


def nvfp4_row_scale(amax: float) -> float:
    """The smallest power of two g >= 2^-126 with amax <= 6 * 448 * g."""
    if not (amax > 0.0) or not math.isfinite(amax):
        return 1.0
    k = max(math.ceil(math.log2(amax / 2688.0)), -126)
    while k > -126 and amax <= 2688.0 * 2.0 ** (k - 1):   # exact comparisons settle the log's rounding
        k -= 1
    while amax > 2688.0 * 2.0 ** k:
        k += 1
    return 2.0 ** k


def nvfp4_block_scale(bamax, g):
    """The smallest positive E4M3 value s with bamax <= 6 g s (1 for a zero
    block); elementwise over arrays of block maxima and row scales."""
    bamax = np.asarray(bamax, dtype=np.float64)
    six_g = 6.0 * np.asarray(g, dtype=np.float64)
    i = np.clip(np.searchsorted(_E4M3_POS, bamax / six_g, side="left"), 1, 126)
    # the quotient may round; the comparisons below are exact and settle it
    i = np.where(six_g * _E4M3_POS[i] < bamax, np.minimum(i + 1, 126), i)
    i = np.where((i > 1) & (six_g * _E4M3_POS[i - 1] >= bamax), i - 1, i)
    return np.where(bamax > 0.0, _E4M3_POS[i], 1.0)


def quantize_nvfp4_act_rows(V: np.ndarray) -> np.ndarray:
    """Each row v -> g s E2M1(v / (g s)) with its row scale g and the block
    scale s of each 16 consecutive elements (the row length is a multiple
    of 16)."""
    V = np.asarray(V, dtype=np.float64)
    R, W = V.shape
    if R == 0 or W == 0:
        return V.copy()
    g = np.array([nvfp4_row_scale(float(a)) for a in np.max(np.abs(V), axis=1)])[:, None]
    B = V.reshape(R, W // 16, 16)
    sc = (nvfp4_block_scale(np.max(np.abs(B), axis=2), g) * g)[:, :, None]
    return (encode_e2m1(B / sc) * sc).reshape(R, W)


def round_bf16(v: np.ndarray) -> np.ndarray:
    """float64 -> nearest fp32 -> nearest bf16 (ties to even), as float64."""
    f = np.asarray(v, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = ((u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000).astype(np.uint32)
    return u.view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------
# Expert FFN (SwiGLU), shared expert, combine
# --------------------------------------------------------------------------


def silu(z: np.ndarray) -> np.ndarray:
    return z / (1.0 + np.exp(-z))


def swiglu_ffn(X: np.ndarray, W13: np.ndarray, W2: np.ndarray, act: Optional[str] = None) -> np.ndarray:
    """O = (silu(X Wg^T) * (X Wu^T)) W2^T with W13 = [Wg; Wu] ([2f, d]) and
    W2 [d, f].  act = "e4m3" / "nvfp4": the rows of X, and of H after
    rounding to bf16, go through quantize_act_rows / quantize_nvfp4_act_rows
    first."""
    f = W2.shape[1]
    quant = {"e4m3": quantize_act_rows, "nvfp4": quantize_nvfp4_act_rows}
    if act is not None and act not in quant:
        raise ValueError(act)
    if act is not None:
        X = quant[act](X)
    G = X @ W13[:f].T
    U = X @ W13[f:].T
    H = silu(G) * U
    if act is not None:
        H = quant[act](round_bf16(H))
    return H @ W2.T


def expert_weights(inp, e: int):
    """Dequantised (W13_e, W2_e) of routed expert e, float64."""
    wd = inp.cfg.w_dtype
    g13 = None if inp.w13_gscale is None else inp.w13_gscale[e]
    g2 = None if inp.w2_gscale is None else inp.w2_gscale[e]
    W13 = dequant(wd, inp.w13[e], None if inp.w13_scale is None else inp.w13_scale[e], g13)
    W2 = dequant(wd, inp.w2[e], None if inp.w2_scale is None else inp.w2_scale[e], g2)
    return W13, W2


def shared_weights(inp):
    wd = inp.cfg.w_dtype
    g13 = None if inp.s13_gscale is None else inp.s13_gscale[0]
    g2 = None if inp.s2_gscale is None else inp.s2_gscale[0]
    W13 = dequant(wd, inp.s13[0], None if inp.s13_scale is None else inp.s13_scale[0], g13)
    W2 = dequant(wd, inp.s2[0], None if inp.s2_scale is None else inp.s2_scale[0], g2)
    return W13, W2


def x_values(inp) -> np.ndarray:
    if inp.cfg.x_dtype == "bf16":
        return decode_bf16(inp.x)
    return np.asarray(inp.x, dtype=np.float64)


def layer_forward(inp, want_intermediates: bool = True, act: Optional[str] = None) -> Dict[str, np.ndarray]:
    """Full layer on all T tokens.

    Returns y [T,d] = shared(x) + sum_j w[t,j] * FFN_{ids[t,j]}(x[t]), with the
    routed terms added in slot order j = 0..k-1, plus the routing outputs and
    (optionally) out_perm (the gate-weighted expert outputs in sorted-pair
    order) and the shared-expert output.
    """
    cfg = inp.cfg
    x = x_values(inp)
    L, ids, w = route(x, inp.w_router, inp.bias, cfg.k)
    counts, offsets, sorted_pair, row_of = permute(ids, cfg.E)
    P = cfg.T * cfg.k
    out_perm = np.zeros((P, cfg.d), dtype=np.float64)
    wflat = w.reshape(-1)
    for e in range(cfg.E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if a == b:
            continue
        pairs = sorted_pair[a:b]
        tok = pairs // cfg.k
        W13, W2 = expert_weights(inp, e)
        out_perm[a:b] = wflat[pairs][:, None] * swiglu_ffn(x[tok], W13, W2, act)
    S13, S2 = shared_weights(inp)
    shared = swiglu_ffn(x, S13, S2, act)
    y = shared.copy()
    for j in range(cfg.k):
        y += out_perm[row_of.reshape(cfg.T, cfg.k)[:, j]]
    res = dict(y=y, logits=L, ids=ids, w=w, counts=counts, offsets=offsets,
               sorted_pair=sorted_pair, row_of=row_of)
    if want_intermediates:
        res.update(out_perm=out_perm, shared=shared)
    return res


def layer_forward_tokens(inp, tokens: Iterable[int], ids_override: Optional[np.ndarray] = None,
                         act: Optional[str] = None):
    """y for a subset of tokens only (sampled checks at full size).

    Routing is computed for the listed tokens; each needed expert is
    dequantised once and applied to just the tokens that picked it.
    ids_override (rows aligned with `tokens`) replaces the selection while the
    gates are still taken from the oracle's own logits.
    """
    cfg = inp.cfg
    tokens = np.asarray(list(tokens), dtype=np.int64)
    x = x_values(inp)[tokens]
    L = router_logits(x, inp.w_router, inp.bias)
    ids = topk_ids(L, cfg.k) if ids_override is None else np.asarray(ids_override, np.int32)
    w = gates(L, ids)
    S13, S2 = shared_weights(inp)
    y = swiglu_ffn(x, S13, S2, act)
    contrib = np.zeros((len(tokens), cfg.k, cfg.d), dtype=np.float64)
    for e in np.unique(ids):
        rows, slots = np.nonzero(ids == e)
        W13, W2 = expert_weights(inp, int(e))
        contrib[rows, slots] = w[rows, slots][:, None] * swiglu_ffn(x[rows], W13, W2, act)
    for j in range(cfg.k):
        y += contrib[:, j]
    return dict(y=y, logits=L, ids=ids, w=w)
