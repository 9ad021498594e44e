"""CPU oracle for the forward of the routed FP8 Mixture-of-Experts FFN layer.

TEST INFRASTRUCTURE ONLY. This module is the slow, plain definition that the
CUDA path is checked against. Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s cpu_baseline / reference legs may import or call it; the product
path never does. It shares no code with the CUDA library and imports nothing
from it: its only shared dependency is the seeded input generator
(``moe_synth``), which holds none of the layer's arithmetic.

Precision: fp64 NumPy for every floating-point step, except where the layer
fixes fp32 (the 1x128 activation quantiser: fp32 scale = amax/448 and an fp32
division before the e4m3 rounding), so that quantised codes are decided in the
same precision as the kernels.

What it computes, and where each step comes from:

* Router ("Kimi-K2-Base", Mixture of experts: Router score = sigmoid over the
  logits of the bf16 gate; "Kimi K2 · Architecture", Weights: the router is
  kept in bfloat16).
* Selection on bias-corrected scores ("Kimi-K2-Base", Mixture of experts:
  Load balancing, e_score_correction_bias added to the sigmoid scores for the
  top-k choice only; Group-limited routing none, n_group = topk_group = 1).
* Weights: the selected experts' unbiased scores, renormalised to sum to 1 and
  then multiplied by the routed scaling factor 2.827 ("Kimi-K2-Base", Mixture
  of experts: Routed scaling factor and Renormalize top-k).
* Experts: SwiGLU, down(silu(gate x) * up x), no bias ("Kimi-K2-Base",
  Feed-forward: Activation and FFN bias); 384 routed plus 1 shared expert of
  2048 hidden features ("Kimi K2 · Architecture", Fact sheet: Feed-forward).
* FP8: e4m3 weights with one fp32 scale per 128x128 block ("Kimi K2 ·
  Architecture", config.json quantization_config), activations quantised
  dynamically in 1x128 groups with fp32 scales ("Kimi-K2-Base", Pretraining
  recipe: Training precision), scale = amax / 448.
* Combine: y = shared(x) + sum_j w_j * expert_{I_j}(x).
* Around the FFN ("Kimi K2 · Dense transformer block", Sources; "Kimi-K2-Base",
  Normalization and stability): the post-attention RMSNorm (eps 1e-6) that
  produces the layer input, and the residual addition after it, followed by the
  next block's input RMSNorm.

Parity pins for every function live in ``tests/test_oracle_*.py``. The layer
output as a whole has no worked example on the pages: its end-to-end value is
pinned only through its parts and through closed-form special cases
(identical experts, selection matrices, integer-exact products).
"""
from __future__ import annotations

import numpy as np

BLOCK = 128
E4M3_MAX = 448.0


# ---------------------------------------------------------------------------
# e4m3 codec, from the OCP 8-bit floating point definition of E4M3:
# 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent field 0
# encodes subnormals (mantissa/8 * 2^-6); no infinities; S.1111.111 is NaN,
# so the largest finite magnitude is S.1111.110 = 1.75 * 2^8 = 448.
# ---------------------------------------------------------------------------

def e4m3_value(code: int) -> float:
    """Value of one e4m3 code, written out from the format's definition."""
    sign = -1.0 if (code >> 7) & 1 else 1.0
    exp = (code >> 3) & 0xF
    man = code & 0x7
    if exp == 0xF and man == 0x7:
        return float("nan")
    if exp == 0:
        return sign * (man / 8.0) * 2.0 ** (1 - 7)
    return sign * (1.0 + man / 8.0) * 2.0 ** (exp - 7)


_DECODE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)
# magnitudes of the positive finite codes 0x00..0x7E; increasing in the code
_POS = _DECODE[:0x7F].copy()


def e4m3_decode(q: np.ndarray) -> np.ndarray:
    """uint8 codes -> fp64 values."""
    return _DECODE[np.asarray(q, dtype=np.uint8)]


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    """Round to the nearest e4m3 value, ties to the even code, saturating to +-448.

    The input is taken at its exact value (fp32 inputs are exact in fp64).
    NaN maps to the NaN code; the sign bit is kept, so -0.0 gives 0x80.
    """
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    nan = np.isnan(a)
    a = np.where(nan, 0.0, a)
    hi = np.searchsorted(_POS, a, side="left")          # _POS[hi-1] < a <= _POS[hi]
    hi = np.minimum(hi, 0x7E)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - _POS[lo]
    d_hi = _POS[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(a >= _POS[0x7E], 0x7E, code)        # saturate to 448
    code = np.where(a == 0.0, 0, code)
    code = code | np.where(np.signbit(v), 0x80, 0)
    code = np.where(nan, 0x7F | np.where(np.signbit(v), 0x80, 0), code)
    return code.astype(np.uint8)


# ---------------------------------------------------------------------------
# 1x128 dynamic activation quantisation (scale = amax / 448, fp32)
# ---------------------------------------------------------------------------

def quantize_1x128(a: np.ndarray):
    """Quantise an fp32 matrix [rows, cols] in groups of 128 consecutive columns.

    Per group: s = fp32(amax) / 448 (fp32 IEEE division); q = e4m3(fp32(a) / s)
    (fp32 IEEE division, then nearest-even rounding with saturation). A group
    whose amax is 0 gets s = 0 and all codes 0x00.
    Returns (q uint8 [rows, cols], s fp32 [rows, cols/128]).
    """
    a = np.ascontiguousarray(a, dtype=np.float32)
    rows, cols = a.shape
    assert cols % BLOCK == 0
    g = a.reshape(rows, cols // BLOCK, BLOCK)
    amax = np.abs(g).max(axis=2)                        # exact in fp32
    s = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    zero = amax == 0
    s_div = np.where(zero, np.float32(1.0), s).astype(np.float32)
    ratio = (g / s_div[:, :, None]).astype(np.float32)  # fp32 division
    q = e4m3_encode(ratio)
    q[np.broadcast_to(zero[:, :, None], q.shape)] = 0
    return q.reshape(rows, cols), s


def dequantize_1x128(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """codes [rows, cols] and scales [rows, cols/128] -> fp64 values."""
    rows, cols = q.shape
    v = e4m3_decode(q).reshape(rows, cols // BLOCK, BLOCK)
    return (v * s.astype(np.float64)[:, :, None]).reshape(rows, cols)


def decode_block_weight(wq: np.ndarray, ws: np.ndarray) -> np.ndarray:
    """e4m3 weight [R, C] with fp32 scales [R/128, C/128] -> fp64 [R, C]."""
    R, C = wq.shape
    v = e4m3_decode(wq).reshape(R // BLOCK, BLOCK, C // BLOCK, BLOCK)
    return (v * ws.astype(np.float64)[:, None, :, None]).reshape(R, C)


# ---------------------------------------------------------------------------
# Router: sigmoid scores, biased top-k choice, renormalised scaled weights
# ---------------------------------------------------------------------------

def router_logits(x: np.ndarray, w_gate: np.ndarray) -> np.ndarray:
    """l = x W_g^T in fp64 over the bf16 values of x [T, d] and W_g [E, d]."""
    return np.asarray(x, np.float64) @ np.asarray(w_gate, np.float64).T


def sigmoid(l: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-l))


def topk_select(c: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest entries per row of c [T, E], in descending order
    of c, equal values ordered by the lower expert id."""
    T, E = c.shape
    out = np.empty((T, k), dtype=np.int32)
    ids = np.arange(E)
    for t in range(T):
        order = np.lexsort((ids, -c[t]))     # primary: -c ascending; then id ascending
        out[t] = order[:k]
    return out


def route(x, w_gate, bias, topk: int, route_scale: float):
    """The gate of one MoE layer.

    Returns a dict with
      scores  fp64 [T, E]  sigmoid(x W_g^T)
      choice  fp64 [T, E]  scores + bias (used only to choose)
      idx     int32 [T, k] chosen experts, descending choice score
      w       fp64 [T, k]  scores[idx] / sum(scores[idx]) * route_scale
      gap     fp64 [T]     choice score of the k-th pick minus the (k+1)-th best
    """
    s = sigmoid(router_logits(x, w_gate))
    c = s + np.asarray(bias, np.float64)[None, :]
    idx = topk_select(c, topk)
    sel = np.take_along_axis(s, idx, axis=1)
    w = sel / sel.sum(axis=1, keepdims=True) * route_scale
    srt = -np.sort(-c, axis=1)
    gap = srt[:, topk - 1] - srt[:, topk] if c.shape[1] > topk else np.full(c.shape[0], np.inf)
    return {"scores": s, "choice": c, "idx": idx, "w": w, "gap": gap}


# ---------------------------------------------------------------------------
# Token permutation into contiguous per-expert segments
# ---------------------------------------------------------------------------

def permute(idx: np.ndarray, E: int):
    """Group the (token, slot) assignments by expert.

    counts[e]    number of tokens that chose expert e
    offsets[e]   exclusive prefix sum of counts over e = 0..E-1; offsets[E] = T*k
    sorted_tok   token ids, segment e = offsets[e]:offsets[e+1], ascending token id
    inv_pos[t,j] position in sorted_tok of the assignment (t, idx[t, j])
    """
    idx = np.asarray(idx)
    T, k = idx.shape
    counts = np.zeros(E, dtype=np.int64)
    sorted_tok = np.empty(T * k, dtype=np.int32)
    inv_pos = np.full((T, k), -1, dtype=np.int32)
    pos = 0
    for e in range(E):
        hit_t, hit_j = np.nonzero(idx == e)          # row-major: ascending token id
        n = hit_t.size
        counts[e] = n
        sorted_tok[pos:pos + n] = hit_t
        inv_pos[hit_t, hit_j] = np.arange(pos, pos + n)
        pos += n
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    return {"counts": counts.astype(np.int32), "offsets": offsets,
            "sorted_tok": sorted_tok, "inv_pos": inv_pos}


# ---------------------------------------------------------------------------
# SwiGLU expert over FP8 weights and quantised activations
# ---------------------------------------------------------------------------

def silu(g: np.ndarray) -> np.ndarray:
    return g / (1.0 + np.exp(-g))


def swiglu_fp8(xq, xs, w1q, w1s, w3q, w3s, w2q, w2s):
    """down(silu(gate x) * up x) for rows of quantised activations.

    xq/xs: e4m3 codes [n, d] and 1x128 scales [n, d/128] of the input rows.
    w1 (gate_proj) and w3 (up_proj): [H, d]; w2 (down_proj): [d, H]; each with
    128x128 block scales. h = silu(g) * u is rounded to fp32 and quantised 1x128
    before the down projection. Returns (o fp64 [n, d], hq, hs).
    """
    h = swiglu_h(xq, xs, w1q, w1s, w3q, w3s)
    hq, hs = quantize_1x128(h)
    o = dequantize_1x128(hq, hs) @ decode_block_weight(w2q, w2s).T
    return o, hq, hs


def swiglu_h(xq, xs, w1q, w1s, w3q, w3s):
    """h = silu(gate x) * up x for rows of quantised activations, formed in fp64
    and rounded to fp32: the value the 1x128 quantiser of the down input sees."""
    xh = dequantize_1x128(xq, xs)
    g = xh @ decode_block_weight(w1q, w1s).T
    u = xh @ decode_block_weight(w3q, w3s).T
    return (silu(g) * u).astype(np.float32)


def _np(t):
    """torch tensor or array -> numpy array (bf16 is widened exactly to fp32)."""
    if hasattr(t, "detach"):
        t = t.detach().cpu()
        if str(t.dtype) == "torch.bfloat16":
            t = t.float()
        return t.numpy()
    return np.asarray(t)


def moe_layer(x, w_gate, bias, experts, topk: int, route_scale: float, n_shared: int = 1,
              tokens=None, idx_override=None):
    """Forward of one routed MoE FFN layer.

    x [T, d] (bf16 values), w_gate [E, d] (bf16 values), bias [E];
    ``experts`` holds w13 [E+S, 2, H, d], w13_s, w2 [E+S, d, H], w2_s as in
    ``moe_synth.ExpertWeights`` (routed experts first, then the shared ones).

    Routing and permutation cover all T tokens. The expert math runs for the
    token ids in ``tokens`` (all tokens when None); y rows of other tokens are
    NaN. ``idx_override`` [T, k] replaces the chosen experts (used to evaluate a
    near-tie token with another valid top-k set); weights are then recomputed
    from the same scores.
    Returns a dict with the route() and permute() fields plus
      xq, xs   the quantised input (all tokens)
      y        fp64 [T, d]
    """
    x = _np(x).astype(np.float32)
    wg = _np(w_gate).astype(np.float32)
    b = _np(bias).astype(np.float64)
    T, d = x.shape
    E = wg.shape[0]
    r = route(x, wg, b, topk, route_scale)
    if idx_override is not None:
        idx = np.asarray(idx_override, dtype=np.int32)
        sel = np.take_along_axis(r["scores"], idx, axis=1)
        r["idx"] = idx
        r["w"] = sel / sel.sum(axis=1, keepdims=True) * route_scale
    p = permute(r["idx"], E)
    xq, xs = quantize_1x128(x)
    toks = np.arange(T) if tokens is None else np.asarray(sorted(set(int(t) for t in tokens)))
    y = np.full((T, d), np.nan)
    y[toks] = 0.0
    w13, w13s, w2, w2s = (_np(experts.w13), _np(experts.w13_s), _np(experts.w2), _np(experts.w2_s))
    wanted = np.zeros(T, dtype=bool)
    wanted[toks] = True
    for e in range(E):
        rows_t = np.nonzero((r["idx"] == e).any(axis=1) & wanted)[0]
        if rows_t.size == 0:
            continue
        o, _, _ = swiglu_fp8(xq[rows_t], xs[rows_t], w13[e, 0], w13s[e, 0], w13[e, 1], w13s[e, 1],
                             w2[e], w2s[e])
        j = np.argmax(r["idx"][rows_t] == e, axis=1)
        y[rows_t] += r["w"][rows_t, j][:, None] * o
    for sidx in range(n_shared):
        e = E + sidx
        o, _, _ = swiglu_fp8(xq[toks], xs[toks], w13[e, 0], w13s[e, 0], w13[e, 1], w13s[e, 1],
                             w2[e], w2s[e])
        y[toks] += o
    out = dict(r)
    out.update(p)
    out.update({"xq": xq, "xs": xs, "y": y, "tokens": toks})
    return out


def dense_swiglu(x, w13, w13_s, w2, w2_s, tokens=None):
    """The dense block's SwiGLU FFN over FP8 weights ("Kimi K2 · Dense transformer
    block", Parameters: SwiGLU MLP). w13 [2, H, d], w2 [d, H] with block scales.
    Returns y fp64 [len(tokens), d] (all tokens when None) and the token ids."""
    x = _np(x).astype(np.float32)
    toks = np.arange(x.shape[0]) if tokens is None else np.asarray(tokens)
    w13, w13s, w2, w2s = _np(w13), _np(w13_s), _np(w2), _np(w2_s)
    xq, xs = quantize_1x128(x[toks])
    o, _, _ = swiglu_fp8(xq, xs, w13[0], w13s[0], w13[1], w13s[1], w2, w2s)
    return o, toks


# ---------------------------------------------------------------------------
# The block around the FFN: RMSNorm and the residual addition
# ---------------------------------------------------------------------------

RMS_NORM_EPS = 1e-6   # "Kimi-K2-Base", Normalization and stability: Norm epsilon


def round_bf16(v: np.ndarray) -> np.ndarray:
    """Round fp64 values to the nearest bfloat16 value (8 significant bits), ties
    to the even significand, in one step from the exact value. Returned as fp64."""
    v = np.asarray(v, dtype=np.float64)
    m, e = np.frexp(v)                       # v = m * 2**e with 0.5 <= |m| < 1
    return np.ldexp(np.rint(m * 256.0) / 256.0, e)   # np.rint: half to even


def rms_norm(h, gamma, eps: float = RMS_NORM_EPS) -> np.ndarray:
    """RMSNorm of each row of h [T, d] with the per-feature weight gamma [d]:
    y = gamma * h / sqrt(mean(h^2) + eps), in fp64 over the bf16 values of h and
    gamma, rounded once to bf16 ("Kimi-K2-Base", Normalization and stability:
    Norm RMSNorm, placement pre, epsilon 1e-06; "Kimi K2 · Dense transformer
    block", Parameters: one 7,168-weight RMSNorm before the attention and one
    before the MLP). Returns fp64 values that are bf16 numbers."""
    h = _np(h).astype(np.float64)
    g = _np(gamma).astype(np.float64)
    inv = 1.0 / np.sqrt((h * h).mean(axis=1, keepdims=True) + eps)
    return round_bf16(h * inv * g)


def residual_add(residual, y) -> np.ndarray:
    """The block's second residual addition, h_next = residual + mlp(x), on bf16
    tensors: the FFN output is a bf16 tensor (y rounded to bf16 first) and the
    sum of the two bf16 values is rounded to bf16 ("Kimi K2 · Dense transformer
    block", Sources: the block's forward adds the residual after the MLP)."""
    r = _np(residual).astype(np.float64)
    return round_bf16(r + round_bf16(_np(y).astype(np.float64)))


def moe_block_ffn(h, gamma_post, w_gate, bias, experts, topk: int, route_scale: float,
                  gamma_next=None, eps: float = RMS_NORM_EPS, n_shared: int = 1,
                  tokens=None, idx_override=None):
    """The FFN half of a MoE block: x = RMSNorm_post(h), y = moe_layer(x),
    h_next = h + y, and, when gamma_next is given, the next block's normalised
    input RMSNorm_next(h_next) ("Kimi K2 · Dense transformer block", Sources:
    residual = h; h = post_attention_layernorm(h); h = mlp(h); h = residual + h;
    the next block starts with its input_layernorm).
    Returns the moe_layer() dict plus x (bf16 values, all tokens), h_next and
    x_next (rows of ``tokens``; other rows NaN)."""
    h = _np(h).astype(np.float32)
    x = rms_norm(h, gamma_post, eps).astype(np.float32)
    out = moe_layer(x, w_gate, bias, experts, topk, route_scale, n_shared=n_shared, tokens=tokens,
                    idx_override=idx_override)
    toks = out["tokens"]
    h_next = np.full(h.shape, np.nan)
    h_next[toks] = residual_add(h[toks], out["y"][toks])
    out["x"] = x
    out["h_next"] = h_next
    if gamma_next is not None:
        x_next = np.full(h.shape, np.nan)
        x_next[toks] = rms_norm(h_next[toks], gamma_next, eps)
        out["x_next"] = x_next
    return out


# ---------------------------------------------------------------------------
# Parameter arithmetic of the layer (pinned against the pages' counts)
# ---------------------------------------------------------------------------

def swiglu_params(d: int, H: int) -> int:
    """gate_proj, up_proj [H, d] and down_proj [d, H], no bias."""
    return 3 * d * H


def moe_layer_params(d: int, E: int, H: int, n_shared: int) -> int:
    """Routed and shared experts, the gate weight [E, d] and the selection bias [E]."""
    return (E + n_shared) * swiglu_params(d, H) + E * d + E
