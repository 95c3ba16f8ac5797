"""CPU oracle for one low-batch MoE decode step -- TEST INFRASTRUCTURE ONLY.

Only the tests, the package smoke check and the benchmark's CPU-baseline leg may
import this module.  The product path (the CUDA library and its binding) never
imports, calls or links it, and shares no code, table or helper with it.

It is a plain, slow, obviously-correct restatement of what the decode step
computes, written from the vLLM API pages on the specialized decode executor:

  [decode page]  vllm.models.glm5next.nvidia.specialized_decode.runtime.decode
                 (class LayerStages: _build_mega, _mega_moe, _router)
  [draft page]   vllm.models.glm5next.nvidia.specialized_decode.runtime.draft
                 (class SpecializedDraft: reduced_norm, run; module docstring)

The pages name the switches of the method but never write its formulas out;
the formulas below are the workload definition the pages' switches imply
(sigmoid scoring, top-k, normalised weights times routed_scaling_factor,
SwiGLU with silu(min(g, L)) * clamp(u, -L, L), RMSNorm with eps inside the
square root).  Every reading taken where the pages are silent is listed in the
repository's design notes and repeated at the function that takes it.

Precision: float64 throughout, except where floating point decides an integer
(an FP8 code, a top-k choice).  The method is stated in fp32; float64 is read
as "no coarser than fp32": every sum the oracle forms is at least as exact as
an fp32 one, so the gap to the GPU path is the GPU's own rounding.  The
integer-deciding steps are taken in float32, the precision the kernels take
them in:
  * router logits are rounded to float32 before scoring, and the selection
    value is sigmoid rounded to float32 plus the float32 bias;
  * activation quantisation (scale = amax / 448, code = RNE_sat(v / scale))
    runs in float32 on float32 values.

Parity pins (tests/test_oracle.py): the FP8 codec is checked exhaustively
against the E4M3 format definition; top-k against brute force over all
subsets; routing weights against their sum invariants; route order against a
brute-force stable sort; RMSNorm against unit RMS; the expert MLP against an
exact int64 matmul (unit scales, integer activations), against a plain
SwiGLU library routine with the limit at infinity, and against a dense average
MLP when k = E with equal scores; the split-K GEMM against a float64 matmul;
the MTP front's concatenation order and normalisation through projections
that select one half (unit RMS of the selected half, the gathered row); the
finalize's slot-to-row pairing through one-hot rows with distinct weights,
and the routed scaling through the linearity of the routed part of m; the
tensor-parallel shards through their sum, which must equal the whole layer's
m (and their h, the matching slices of the whole layer's h).
The full layer on real shapes is pinned only through these pieces.
"""

from __future__ import annotations

import math

import numpy as np

QMAX = 448.0  # largest finite E4M3 magnitude (1.75 * 2^8)
BLOCK = 128  # side of a weight scale block and length of an activation group


# --------------------------------------------------------------------------
# FP8 E4M3 codec, from the format definition (1 sign, 4 exponent bits with
# bias 7, 3 mantissa bits; no infinities; S.1111.111 is NaN; exponent field 0
# holds subnormals m/8 * 2^-6).
# --------------------------------------------------------------------------

def _build_e4m3_table() -> np.ndarray:
    vals = np.empty(256, np.float64)
    for c in range(256):
        sign = -1.0 if c & 0x80 else 1.0
        e = (c >> 3) & 0xF
        m = c & 0x7
        if e == 0xF and m == 0x7:
            vals[c] = np.nan
        elif e == 0:
            vals[c] = sign * (m / 8.0) * 2.0 ** -6
        else:
            vals[c] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


E4M3_VALUES = _build_e4m3_table()
# codes 0x00..0x7E are the non-negative finite values in increasing order
_POS = E4M3_VALUES[:127].copy()


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """Value (float64) of each E4M3 code."""
    return E4M3_VALUES[np.asarray(codes, np.uint8)]


def e4m3_encode(v) -> np.ndarray:
    """Round float32 values to E4M3 codes: nearest, ties to even mantissa,
    saturating to +-448 (the 'satfinite' rounding).  NaN is not expected."""
    v = np.asarray(v, np.float32).astype(np.float64)
    mag = np.minimum(np.abs(v), QMAX)
    hi = np.clip(np.searchsorted(_POS, mag, side="left"), 0, 126)
    lo = np.maximum(hi - 1, 0)
    d_lo = mag - _POS[lo]
    d_hi = _POS[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    sign = np.signbit(v).astype(np.uint8) << 7
    return code | sign


def bf16_round(v) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 (ties to even), once,
    returned as float64.  Normal range only (no overflow in this workload)."""
    v = np.asarray(v, np.float64)
    m, e = np.frexp(v)  # v = m * 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.round(np.ldexp(m, 8)), e - 8)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Value of bfloat16 numbers given as their uint16 bit patterns."""
    b = np.asarray(bits, np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------
# Block scales
# --------------------------------------------------------------------------

def pow2_round_up(s: np.ndarray) -> np.ndarray:
    """e8m0 reading of a float32 scale: the smallest power of two >= s."""
    s = np.asarray(s, np.float32)
    m, e = np.frexp(s)
    up = np.ldexp(np.float32(1.0), e).astype(np.float32)
    return np.where(m == 0.5, s, up).astype(np.float32)


def dequant_weight(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """w[r, c] = E4M3(codes[r, c]) * scales[r // 128, c // 128] (float64).

    The weights and their *_scale_inv tensors of the [decode page],
    LayerStages._build_mega: the scale multiplies the code."""
    w = e4m3_decode(codes)
    s = np.repeat(np.repeat(np.asarray(scales, np.float64), BLOCK, 0), BLOCK, 1)
    return w * s[: w.shape[0], : w.shape[1]]


def quantize_act(v32: np.ndarray, e8m0: bool):
    """Per-row, per-128-column-group FP8 quantisation of float32 activations.

    scale = amax / 448 in float32 (a power of two rounded up when e8m0), 1 when
    the group is all zero; code = RNE_sat(v / scale) with the division in
    float32.  Returns (codes uint8 [n, K], scales float32 [n, K/128])."""
    v32 = np.asarray(v32, np.float32)
    n, K = v32.shape
    g = v32.reshape(n, K // BLOCK, BLOCK)
    amax = np.abs(g).max(axis=2)
    scale = (amax / np.float32(QMAX)).astype(np.float32)
    if e8m0:
        scale = pow2_round_up(scale)
    scale = np.where(amax == 0, np.float32(1.0), scale).astype(np.float32)
    q = (g / scale[:, :, None]).astype(np.float32)
    return e4m3_encode(q).reshape(n, K), scale


def dequant_act(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    n, K = codes.shape
    v = e4m3_decode(codes).reshape(n, K // BLOCK, BLOCK)
    return (v * np.asarray(scales, np.float64)[:, :, None]).reshape(n, K)


# --------------------------------------------------------------------------
# Router: logits, sigmoid scoring, top-k, normalised scaled weights
# ([decode page], LayerStages._build_mega accepts only sigmoid scoring with
# n_group == 1 and norm_topk_prob; _mega_moe passes e_score_correction_bias;
# _router computes fp32 logits from the bf16 gate weight).
# --------------------------------------------------------------------------

def router_logits(x: np.ndarray, w_router: np.ndarray) -> np.ndarray:
    """logits[t, e] = sum_h x[t, h] * W[e, h], float64 then rounded to float32
    (the gate's output dtype)."""
    return (np.asarray(x, np.float64) @ np.asarray(w_router, np.float64).T).astype(np.float32)


def sigmoid_scores(logits32: np.ndarray) -> np.ndarray:
    """s = 1 / (1 + exp(-logit)), evaluated in float64, rounded to float32."""
    l = np.asarray(logits32, np.float64)
    return (1.0 / (1.0 + np.exp(-l))).astype(np.float32)


def selection_values(scores32: np.ndarray, bias) -> np.ndarray:
    """Selection value: score plus the per-expert correction bias (float32)."""
    if bias is None:
        return scores32.astype(np.float32)
    return (scores32 + np.asarray(bias, np.float32)[None, :]).astype(np.float32)


def topk_select(sel: np.ndarray, k: int) -> np.ndarray:
    """ids[t, j]: the k experts with the largest selection value, in
    descending order of that value; an exact tie goes to the lower id."""
    M, E = sel.shape
    ids = np.empty((M, k), np.int32)
    for t in range(M):
        order = sorted(range(E), key=lambda e: (-float(sel[t, e]), e))
        ids[t] = order[:k]
    return ids


def routing_weights(scores32: np.ndarray, ids: np.ndarray, routed_scaling: float) -> np.ndarray:
    """w[t, j] = s[t, id_j] / sum_j s[t, id_j] * routed_scaling (float64).
    The weights use the unbiased scores; the bias only steers selection."""
    s = np.take_along_axis(np.asarray(scores32, np.float64), ids.astype(np.int64), axis=1)
    return s / s.sum(axis=1, keepdims=True) * float(routed_scaling)


def route(x, w_router, bias, k, routed_scaling):
    logits = router_logits(x, w_router)
    scores = sigmoid_scores(logits)
    sel = selection_values(scores, bias)
    ids = topk_select(sel, k)
    w = routing_weights(scores, ids, routed_scaling)
    return logits, scores, sel, ids, w


def route_order(ids: np.ndarray, num_experts: int):
    """Stable counting sort of the expanded route index r = t*k + j by expert
    id.  Returns (sorted_routes int32 [M*k], expert_offsets int32 [E+1]).

    The [decode page] (LayerStages._mega_moe) hands the routed rows over in
    expanded (token-major) order with the identity expanded->permuted map; the
    grouping of routes by expert is the order the expert work runs in."""
    flat = np.asarray(ids, np.int64).reshape(-1)
    sorted_routes = []
    offsets = [0]
    for e in range(num_experts):
        for r in range(flat.size):
            if flat[r] == e:
                sorted_routes.append(r)
        offsets.append(len(sorted_routes))
    return np.asarray(sorted_routes, np.int32), np.asarray(offsets, np.int32)


# --------------------------------------------------------------------------
# Expert MLP: w13 GEMM, clamped SwiGLU, w2 GEMM (FP8 operands, 128x128 scales)
# ([decode page] LayerStages._build_mega: w13_weight, w13_weight_scale_inv,
# w2_weight, w2_weight_scale_inv, swiglu_limit, the e8m0 switch; the shared
# expert takes the same arguments through SharedExpert).
# --------------------------------------------------------------------------

def silu(z):
    return z / (1.0 + np.exp(-z))


def swiglu_clamped(g, u, limit):
    """h = silu(min(g, L)) * clamp(u, -L, L).  Rows [0, I) of w13 give g,
    rows [I, 2I) give u."""
    return silu(np.minimum(g, limit)) * np.clip(u, -limit, limit)


def expert_mlp(xq, xs, w13_deq, w2_deq, limit, e8m0):
    """One expert on n quantised activation rows.

    xq/xs: the rows' FP8 codes and per-128-group scales.  Returns
    (y float64 [n, H], h32 float32 [n, I], hq, hs)."""
    x = dequant_act(xq, xs)
    gu = x @ w13_deq.T
    inter = w13_deq.shape[0] // 2
    h = swiglu_clamped(gu[:, :inter], gu[:, inter:], limit)
    h32 = h.astype(np.float32)
    hq, hs = quantize_act(h32, e8m0)
    y = dequant_act(hq, hs) @ w2_deq.T
    return y, h32, hq, hs


# --------------------------------------------------------------------------
# Boundary: finalize + residual add + RMSNorm ([draft page]: the MTP layer's
# boundary fuses the residual add with the RMSNorm; reduced_norm gives back
# the normalised sum and the updated residual).
# --------------------------------------------------------------------------

def rmsnorm_residual(m, residual_bf16, gain_bf16, eps):
    """r' = m + residual; residual_out = bf16(r'); out = bf16(r'_bf16 *
    1/sqrt(mean(r'_bf16^2) + eps) * gain).  All arguments float64 values."""
    r = np.asarray(m, np.float64) + np.asarray(residual_bf16, np.float64)
    rb = bf16_round(r)
    ms = (rb * rb).mean(axis=1, keepdims=True)
    out = bf16_round(rb / np.sqrt(ms + eps) * np.asarray(gain_bf16, np.float64)[None, :])
    return out, rb


def finalize(rows, w, shared):
    """m[t] = sum_j w[t, j] * rows[t*k + j] + shared[t] (rows in expanded
    order, as handed over by the [decode page]'s UnfinalizedMoEOutput)."""
    M, k = w.shape
    H = rows.shape[1]
    m = np.zeros((M, H), np.float64)
    for t in range(M):
        for j in range(k):
            m[t] += w[t, j] * rows[t * k + j]
    if shared is not None:
        m += shared
    return m


# --------------------------------------------------------------------------
# Whole layer
# --------------------------------------------------------------------------

class Layer:
    """Host copies of one layer's weights, as numpy arrays.

    router_w: bf16 values as float64 [E, H]; sel_bias float32 [E] or None;
    w13 uint8 [E, 2I, H], w13_s float32 [E, 2I/128, H/128];
    w2 uint8 [E, H, I], w2_s float32 [E, H/128, I/128];
    sw13/sw13_s/sw2/sw2_s the shared expert alike (leading dim dropped);
    gain: bf16 values as float64 [H]."""

    def __init__(self, *, router_w, sel_bias, w13, w13_s, w2, w2_s, sw13, sw13_s,
                 sw2, sw2_s, gain, top_k, routed_scaling, swiglu_limit, rms_eps, e8m0,
                 has_shared=None):
        self.router_w = np.asarray(router_w, np.float64)
        self.sel_bias = None if sel_bias is None else np.asarray(sel_bias, np.float32)
        self.w13, self.w13_s, self.w2, self.w2_s = w13, w13_s, w2, w2_s
        self.sw13, self.sw13_s, self.sw2, self.sw2_s = sw13, sw13_s, sw2, sw2_s
        self.gain = np.asarray(gain, np.float64)
        self.top_k = int(top_k)
        self.routed_scaling = float(routed_scaling)
        self.swiglu_limit = float(swiglu_limit)
        self.rms_eps = float(rms_eps)
        self.e8m0 = bool(e8m0)
        # a layer without a shared expert (shared_inter = 0) passes no shared weights
        self.has_shared = (sw13 is not None) if has_shared is None else bool(has_shared)
        self._cache: dict = {}

    @property
    def num_experts(self):
        return self.router_w.shape[0]

    def expert(self, e):
        """Dequantised (w13, w2) of routed expert e, or the shared expert for
        e == -1.  One expert at a time is kept."""
        if e not in self._cache:
            self._cache.clear()
            if e < 0:
                self._cache[e] = (dequant_weight(self.sw13, self.sw13_s),
                                  dequant_weight(self.sw2, self.sw2_s))
            else:
                self._cache[e] = (dequant_weight(self.w13[e], self.w13_s[e]),
                                  dequant_weight(self.w2[e], self.w2_s[e]))
        return self._cache[e]


def moe_decode_layer(layer: Layer, x_bf16, residual_bf16, tokens=None):
    """The decode step: router -> top-k -> route order -> experts (+ shared)
    -> weighted finalize -> residual add -> RMSNorm.

    x_bf16, residual_bf16: float64 values of bf16 inputs [M, H].
    tokens: optional subset of token indices whose outputs are computed (the
    routing is always computed for every token, since route order depends on
    all of them).  Returns a dict of every result and intermediate."""
    M, H = x_bf16.shape
    k = layer.top_k
    E = layer.num_experts
    if E == 0:
        # a dense layer ([decode page] LayerStages._build_dense: a dense MLP as
        # GEMVs, the shared-expert path with no router): no routes at all
        k = 0
        logits = scores = sel = np.zeros((M, 0))
        ids = np.zeros((M, 0), np.int64)
        w = np.zeros((M, 0))
        sorted_routes, offsets = np.zeros(0, np.int64), np.zeros(1, np.int64)
    else:
        logits, scores, sel, ids, w = route(x_bf16, layer.router_w, layer.sel_bias, k,
                                            layer.routed_scaling)
        sorted_routes, offsets = route_order(ids, E)
    if tokens is None:
        tokens = np.arange(M)
    tokens = np.asarray(tokens, np.int64)
    xq, xs = quantize_act(np.asarray(x_bf16, np.float32), layer.e8m0)
    rows = np.zeros((M * k, H), np.float64)
    shared = np.zeros((M, H), np.float64)
    h_rows = {}
    need = set(int(t) for t in tokens)
    for e in range(E):
        rs = [int(r) for r in sorted_routes[offsets[e]:offsets[e + 1]] if int(r) // k in need]
        if not rs:
            continue
        w13d, w2d = layer.expert(e)
        tok = np.asarray([r // k for r in rs])
        y, h32, _, _ = expert_mlp(xq[tok], xs[tok], w13d, w2d, layer.swiglu_limit, layer.e8m0)
        for i, r in enumerate(rs):
            rows[r] = y[i]
            h_rows[r] = h32[i]
    if layer.has_shared:
        w13d, w2d = layer.expert(-1)
        ys, hs32, _, _ = expert_mlp(xq[tokens], xs[tokens], w13d, w2d, layer.swiglu_limit, layer.e8m0)
        shared[tokens] = ys
    m = finalize(rows, w, shared)
    out, res_out = rmsnorm_residual(m[tokens], residual_bf16[tokens], layer.gain, layer.rms_eps)
    return dict(logits=logits, scores=scores, sel=sel, ids=ids, weights=w,
                sorted_routes=sorted_routes, offsets=offsets, xq=xq, xs=xs,
                rows=rows, shared=shared, h_rows=h_rows, m=m, tokens=tokens,
                out=out, residual_out=res_out)


# --------------------------------------------------------------------------
# Tensor parallelism over each expert's intermediate dimension ([decode page]
# LayerStages: the MoE sublayer is left TP-partial; [draft page] module
# docstring: the boundary fuses the all-reduce with the residual add and the
# RMSNorm).  The reading: rank g of G keeps the gate rows [g I/G, (g+1) I/G),
# the same up rows and the same w2 columns of every expert, with their block
# scales (I/G a multiple of 128); the router is replicated.
# --------------------------------------------------------------------------

def tp_shard(layer: Layer, g: int, G: int) -> Layer:
    """Rank g of G's share of a layer (numpy weight arrays)."""
    def w13_rows(codes, scales, a, b):
        inter = codes.shape[-2] // 2
        c = np.concatenate([codes[..., a:b, :], codes[..., inter + a:inter + b, :]], axis=-2)
        s = np.concatenate([scales[..., a // BLOCK:b // BLOCK, :],
                            scales[..., (inter + a) // BLOCK:(inter + b) // BLOCK, :]], axis=-2)
        return c, s

    def w2_cols(codes, scales, a, b):
        return codes[..., a:b], scales[..., a // BLOCK:b // BLOCK]

    def cut(n):
        assert n % (G * BLOCK) == 0, "shards of whole 128-blocks"
        return g * n // G, (g + 1) * n // G

    kw = {}
    if layer.w13 is not None:
        a, b = cut(layer.w13.shape[-2] // 2)
        kw["w13"], kw["w13_s"] = w13_rows(layer.w13, layer.w13_s, a, b)
        kw["w2"], kw["w2_s"] = w2_cols(layer.w2, layer.w2_s, a, b)
    else:
        kw.update(w13=None, w13_s=None, w2=None, w2_s=None)
    if layer.has_shared:
        a, b = cut(layer.sw13.shape[-2] // 2)
        kw["sw13"], kw["sw13_s"] = w13_rows(layer.sw13, layer.sw13_s, a, b)
        kw["sw2"], kw["sw2_s"] = w2_cols(layer.sw2, layer.sw2_s, a, b)
    else:
        kw.update(sw13=None, sw13_s=None, sw2=None, sw2_s=None)
    return Layer(router_w=layer.router_w, sel_bias=layer.sel_bias, gain=layer.gain, top_k=layer.top_k,
                 routed_scaling=layer.routed_scaling, swiglu_limit=layer.swiglu_limit, rms_eps=layer.rms_eps,
                 e8m0=layer.e8m0, has_shared=layer.has_shared, **kw)


def tp_boundary(partials, residual_bf16, gain_bf16, eps):
    """The boundary over the ranks' shares of m: their sum (in rank order),
    then the residual add and RMSNorm of rmsnorm_residual."""
    m = np.zeros_like(np.asarray(partials[0], np.float64))
    for p in partials:
        m = m + np.asarray(p, np.float64)
    return rmsnorm_residual(m, residual_bf16, gain_bf16, eps)


# --------------------------------------------------------------------------
# Split-K BF16 projection ([draft page]: the draft's BF16 projections, such
# as eh_proj, run a split-K GEMM above two tokens).  The split is an
# implementation choice; the result is the plain product.
# --------------------------------------------------------------------------

def projection(a_bf16, w_bf16, alpha=1.0, out_fp32=False):
    """Y[M, N] = alpha * A[M, K] @ W[N, K]^T in float64, rounded to bf16
    (or to float32 for the fp32-output form used by the router)."""
    y = float(alpha) * (np.asarray(a_bf16, np.float64) @ np.asarray(w_bf16, np.float64).T)
    if out_fp32:
        return y.astype(np.float32).astype(np.float64)
    return bf16_round(y)


def rmsnorm(x_bf16, gain_bf16, eps):
    """bf16(x * 1/sqrt(mean(x^2) + eps) * gain), per row; x already bf16 values."""
    x = np.asarray(x_bf16, np.float64)
    ms = (x * x).mean(axis=1, keepdims=True)
    return bf16_round(x / np.sqrt(ms + eps) * np.asarray(gain_bf16, np.float64)[None, :])


def mtp_front(ids, embed_bf16, hidden_bf16, enorm_bf16, hnorm_bf16, eps, eh_w_bf16):
    """The MTP layer's input projection ([draft page] SpecializedDraft.run:
    the embedding of the input tokens and the previous hidden state, each
    RMS-normalised with its own gain (enorm / hnorm, one eps), concatenated and
    projected by eh_proj).  Readings: the embedding half comes first (the name
    eh_proj: e then h); the concatenated input is bf16, as the BF16 split-K
    projection reads it.  Returns (A [M, 2H] bf16 values, Y [M, H] bf16)."""
    ids = np.asarray(ids, np.int64)
    e = np.asarray(embed_bf16, np.float64)[ids]
    a = np.concatenate([rmsnorm(e, enorm_bf16, eps), rmsnorm(hidden_bf16, hnorm_bf16, eps)], axis=1)
    return a, projection(a, eh_w_bf16)


def rms(v):
    v = np.asarray(v, np.float64)
    return math.sqrt(float((v * v).mean())) if v.size else 0.0


def max_abs_rel(got, ref):
    """max_i |got_i - ref_i| / max(|ref_i|, rms(ref)): relative where values
    are large, scaled by the tensor's RMS near zero."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if ref.size == 0:
        return 0.0
    den = np.maximum(np.abs(ref), rms(ref))
    den = np.where(den == 0, 1.0, den)
    return float((np.abs(got - ref) / den).max())
