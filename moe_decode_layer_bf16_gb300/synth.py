"""Seeded synthetic inputs for the MoE decode layer and the split-K projection.

This module only draws random tensors; it holds none of the decode step's
arithmetic.  Both the CUDA path (through the tests and the benchmark) and the
CPU oracle consume what it produces.  Every tensor is drawn from its own
torch.Generator seeded from (seed, tensor tag, expert index), so any one
expert can be regenerated without the others.

Recipe (the shapes and distributions of the workloads the layer is measured
on; the weights are random-init, no trained checkpoint is involved):
  * x, residual ~ N(0, 1) rounded to bf16, [M, H];
  * router weight ~ N(0, router_std) in bf16, [E, H]; router_std defaults to
    0.05 * sqrt(512 / H), which keeps the logit spread of the H = 512 layer;
  * expert w13 [2I, H] and w2 [H, I] drawn N(0, 0.02) in float32 and stored as
    FP8 E4M3 codes with one float32 scale per 128x128 block: the block scale is
    the block's amax / 448 (rounded up to a power of two for the e8m0 form) and
    the code is torch's float8_e4m3fn conversion of weight / scale;
  * the shared expert likewise; the norm gain ~ 1 + N(0, 0.1) in bf16;
  * optional per-expert selection bias ~ N(0, bias_std) in float32;
  * optional Zipf popularity: expert e gets popularity rank rank(e) from a
    seeded permutation, router column 0 is set to -zipf_s * log(rank(e))
    (centred), and token feature 0 is set to 1, so the logit of expert e
    carries that offset for every token;
  * split-K projection: A ~ N(0, 1) and W ~ N(0, 0.02), both bf16.
"""

from __future__ import annotations

import math

import torch

from .dims import LayerDims

_TAGS = {"router": 1, "w13": 2, "w2": 3, "sw13": 4, "sw2": 5, "gain": 6, "bias": 7,
         "x": 8, "residual": 9, "zipf": 10, "proj_a": 11, "proj_w": 12, "token": 13}


def _gen(seed: int, tag: str, index: int, device) -> torch.Generator:
    s = (int(seed) * 1_000_003 + _TAGS[tag] * 7_919 + int(index) * 104_729) & 0x7FFF_FFFF_FFFF
    g = torch.Generator(device=device)
    g.manual_seed(s)
    return g


def _randn(shape, seed, tag, index, device, std=1.0):
    g = _gen(seed, tag, index, device)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std


def fp8_blocks(w32: torch.Tensor, e8m0: bool):
    """Store a float32 [R, C] weight as E4M3 codes (uint8) plus float32
    128x128 block scales [R/128, C/128]."""
    R, C = w32.shape
    b = w32.reshape(R // 128, 128, C // 128, 128)
    amax = b.abs().amax(dim=(1, 3))
    s = amax / 448.0
    if e8m0:
        m, e = torch.frexp(s)
        s = torch.where(m == 0.5, s, torch.ldexp(torch.ones_like(s), e))
    s = torch.where(amax == 0, torch.ones_like(s), s).to(torch.float32)
    q = (b / s[:, None, :, None]).clamp(-448.0, 448.0)
    codes = q.to(torch.float8_e4m3fn).view(torch.uint8).reshape(R, C)
    return codes.contiguous(), s.contiguous()


def make_expert(dims: LayerDims, e: int, seed: int = 0, device="cpu", weight_std: float = 0.02):
    """Routed expert e alone: (w13 codes, w13 scales, w2 codes, w2 scales)."""
    H, I = dims.hidden, dims.inter
    w13, w13_s = fp8_blocks(_randn((2 * I, H), seed, "w13", e, device, weight_std), dims.e8m0)
    w2, w2_s = fp8_blocks(_randn((H, I), seed, "w2", e, device, weight_std), dims.e8m0)
    return w13, w13_s, w2, w2_s


def make_layer(dims: LayerDims, seed: int = 0, device="cpu", router_std=None,
               bias_std: float | None = None, zipf_s: float | None = None,
               weight_std: float = 0.02, experts=None) -> dict:
    """All weights of one layer as torch tensors on `device`.  With `experts`
    given, only those routed experts are drawn (the others are left as zero
    codes with unit scales); experts=[] skips the routed experts' tensors
    altogether (w13, w2 and their scales are then None)."""
    H, I, Is, E = dims.hidden, dims.inter, dims.shared_inter, dims.num_experts
    if router_std is None:
        router_std = 0.05 * math.sqrt(512.0 / H)
    router = _randn((E, H), seed, "router", 0, device, router_std)
    if zipf_s is not None:
        g = _gen(seed, "zipf", 0, "cpu")
        perm = torch.randperm(E, generator=g)
        rank = torch.empty(E, dtype=torch.float64)
        rank[perm] = torch.arange(1, E + 1, dtype=torch.float64)
        off = -float(zipf_s) * torch.log(rank)
        off = off - off.mean()
        router[:, 0] = off.to(torch.float32).to(device)
    if experts is not None and len(experts) == 0:
        w13 = w13_s = w2 = w2_s = None
        experts = []
    else:
        w13 = torch.zeros((E, 2 * I, H), dtype=torch.uint8, device=device)
        w13_s = torch.ones((E, 2 * I // 128, H // 128), dtype=torch.float32, device=device)
        w2 = torch.zeros((E, H, I), dtype=torch.uint8, device=device)
        w2_s = torch.ones((E, H // 128, I // 128), dtype=torch.float32, device=device)
    for e in (range(E) if experts is None else sorted(set(int(v) for v in experts))):
        w13[e], w13_s[e], w2[e], w2_s[e] = make_expert(dims, e, seed, device, weight_std)
    layer = dict(router_w=router.to(torch.bfloat16), w13=w13, w13_s=w13_s, w2=w2, w2_s=w2_s)
    if Is > 0:
        layer["sw13"], layer["sw13_s"] = fp8_blocks(
            _randn((2 * Is, H), seed, "sw13", 0, device, weight_std), dims.e8m0)
        layer["sw2"], layer["sw2_s"] = fp8_blocks(
            _randn((H, Is), seed, "sw2", 0, device, weight_std), dims.e8m0)
    else:
        layer["sw13"] = layer["sw13_s"] = layer["sw2"] = layer["sw2_s"] = None
    layer["gain"] = (1.0 + _randn((H,), seed, "gain", 0, device, 0.1)).to(torch.bfloat16)
    layer["sel_bias"] = (None if bias_std is None
                         else _randn((E,), seed, "bias", 0, device, bias_std).contiguous())
    return layer


def make_tokens(M: int, H: int, seed: int = 0, device="cpu", zipf: bool = False):
    """x and residual, bf16 [M, H]."""
    x = _randn((M, H), seed, "x", 0, device)
    if zipf and M > 0:
        x[:, 0] = 1.0
    res = _randn((M, H), seed, "residual", 0, device)
    return x.to(torch.bfloat16).contiguous(), res.to(torch.bfloat16).contiguous()


def redraw_token(x: torch.Tensor, t: int, seed: int, attempt: int, zipf: bool = False):
    """Replace row t of x by a fresh N(0, 1) draw from a per-token sub-seed."""
    H = x.shape[1]
    row = _randn((H,), seed, "token", (t + 1) * 4096 + attempt, x.device)
    if zipf:
        row[0] = 1.0
    x[t] = row.to(x.dtype)


def make_projection(M: int, N: int, K: int, seed: int = 0, device="cpu"):
    """A bf16 [M, K] ~ N(0, 1), W bf16 [N, K] ~ N(0, 0.02)."""
    a = _randn((M, K), seed, "proj_a", 0, device).to(torch.bfloat16)
    w = _randn((N, K), seed, "proj_w", 0, device, 0.02).to(torch.bfloat16)
    return a.contiguous(), w.contiguous()
