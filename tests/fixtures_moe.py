"""Test-side helpers: seeded layers and tokens, their oracle view, and the
no-near-tie condition on routing.

The routing must be decided identically by the CUDA path (float32 logits
summed in its own order) and the oracle (float64 logits rounded to float32).
Inputs are therefore drawn so that, for every token, the selection values of
the k+1 best experts are pairwise at least `delta` apart (computed in float64
by the oracle); a token that fails is redrawn from a per-token sub-seed.
"""

from __future__ import annotations

import numpy as np
import torch

from moe_decode_layer_bf16_gb300 import synth
from moe_decode_layer_bf16_gb300.dims import LayerDims
from oracle import moe_oracle as orc

DELTA = 1e-4


def to_np(t):
    if t is None:
        return None
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.float().numpy().astype(np.float64)
    return t.numpy()


def oracle_layer(dims: LayerDims, lw: dict) -> orc.Layer:
    return orc.Layer(
        router_w=to_np(lw["router_w"]), sel_bias=to_np(lw["sel_bias"]),
        w13=to_np(lw["w13"]), w13_s=to_np(lw["w13_s"]), w2=to_np(lw["w2"]), w2_s=to_np(lw["w2_s"]),
        sw13=to_np(lw["sw13"]), sw13_s=to_np(lw["sw13_s"]), sw2=to_np(lw["sw2"]), sw2_s=to_np(lw["sw2_s"]),
        gain=to_np(lw["gain"]), top_k=dims.top_k, routed_scaling=dims.routed_scaling,
        swiglu_limit=dims.swiglu_limit, rms_eps=dims.rms_eps, e8m0=dims.e8m0)


def min_gap(x64: np.ndarray, router64: np.ndarray, bias, k: int) -> np.ndarray:
    """Per token: the smallest gap between adjacent selection values among the
    k+1 best experts, in float64."""
    logits = x64 @ router64.T
    s = 1.0 / (1.0 + np.exp(-logits))
    if bias is not None:
        s = s + np.asarray(bias, np.float64)[None, :]
    srt = -np.sort(-s, axis=1)[:, : min(k + 1, s.shape[1])]
    if srt.shape[1] < 2:
        return np.full(s.shape[0], np.inf)
    return np.min(srt[:, :-1] - srt[:, 1:], axis=1)


def tie_free_tokens(dims: LayerDims, lw: dict, M: int, seed: int, zipf: bool = False,
                    delta: float = DELTA, device="cpu"):
    """x, residual (bf16 torch on `device`) with every token's routing margin
    at least `delta`.  Returns (x, residual, number of redrawn rows)."""
    x, res = synth.make_tokens(M, dims.hidden, seed, device=device, zipf=zipf)
    router64 = to_np(lw["router_w"])
    bias = to_np(lw["sel_bias"])
    redrawn = 0
    for attempt in range(50):
        gaps = min_gap(to_np(x), router64, bias, dims.top_k)
        bad = np.nonzero(gaps < delta)[0]
        if bad.size == 0:
            return x, res, redrawn
        for t in bad:
            synth.redraw_token(x, int(t), seed, attempt, zipf=zipf)
            redrawn += 1
    raise RuntimeError("could not draw tie-free tokens")
