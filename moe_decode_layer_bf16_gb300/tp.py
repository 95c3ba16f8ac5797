"""Tensor parallelism over each expert's intermediate dimension: host-side
plumbing around the library's per-rank entry points.

The decode page (vllm.models.glm5next.nvidia.specialized_decode.runtime
.decode, class LayerStages) leaves the MoE sublayer "TP-partial" and the draft
page's module docstring fuses the all-reduce with the residual add and the
RMSNorm at the boundary.  Here rank g of G keeps, of every routed expert and
of the shared expert, the gate rows [g I/G, (g+1) I/G) and the same up rows of
w13 and the same columns of w2, with their 128 x 128 block scales; the router
is replicated, so every rank routes identically.  A shard is an ordinary MoE
layer with inter = I/G and shared_inter = I_s/G, which the library runs with
moe_decode_layer_partial (the rank's fp32 share of m); the shares are summed by
an all-reduce over the ranks and moe_tp_boundary adds the residual and
normalises.

Only slicing and collectives here: the arithmetic is the library's.
"""

from __future__ import annotations

import torch

from .dims import LayerDims

BLOCK = 128


def shard_dims(dims: LayerDims, G: int) -> LayerDims:
    """The layer dimensions of one of G ranks' shards."""
    for what, n in (("inter", dims.inter), ("shared_inter", dims.shared_inter)):
        if n % (G * BLOCK):
            raise ValueError(f"{what} = {n} does not split into {G} shards of whole 128-blocks")
    return dims.with_(inter=dims.inter // G, shared_inter=dims.shared_inter // G)


def _w13_rows(codes, scales, inter, a, b):
    """Gate rows [a, b) and up rows [inter + a, inter + b) of a w13 tensor
    [..., 2 inter, H] and of its block scales [..., 2 inter / 128, H / 128]."""
    c = torch.cat([codes[..., a:b, :], codes[..., inter + a:inter + b, :]], dim=-2).contiguous()
    s = torch.cat([scales[..., a // BLOCK:b // BLOCK, :],
                   scales[..., (inter + a) // BLOCK:(inter + b) // BLOCK, :]], dim=-2).contiguous()
    return c, s


def _w2_cols(codes, scales, a, b):
    """Columns [a, b) of a w2 tensor [..., H, inter] and of its block scales."""
    return codes[..., a:b].contiguous(), scales[..., a // BLOCK:b // BLOCK].contiguous()


def shard_weights(dims: LayerDims, weights: dict, g: int, G: int) -> dict:
    """Rank g of G's weights (new contiguous tensors on the same device); the
    router weight, selection bias and norm gain are shared with the input."""
    if not 0 <= g < G:
        raise ValueError("rank out of range")
    shard_dims(dims, G)
    out = dict(weights)
    I, Is = dims.inter, dims.shared_inter
    if weights.get("w13") is not None:
        a, b = g * I // G, (g + 1) * I // G
        out["w13"], out["w13_s"] = _w13_rows(weights["w13"], weights["w13_s"], I, a, b)
        out["w2"], out["w2_s"] = _w2_cols(weights["w2"], weights["w2_s"], a, b)
    if Is > 0 and weights.get("sw13") is not None:
        a, b = g * Is // G, (g + 1) * Is // G
        out["sw13"], out["sw13_s"] = _w13_rows(weights["sw13"], weights["sw13_s"], Is, a, b)
        out["sw2"], out["sw2_s"] = _w2_cols(weights["sw2"], weights["sw2_s"], a, b)
    return out


def all_reduce_partials(m: torch.Tensor, group=None) -> torch.Tensor:
    """Sum the ranks' shares of m (float32 [M, H]) in place over the process
    group (NCCL on GPUs, gloo on the host); returns m."""
    import torch.distributed as dist
    dist.all_reduce(m, op=dist.ReduceOp.SUM, group=group)
    return m


def tp_decode_layer(dims: LayerDims, shard: dict, x, residual, workspace, out=None, residual_out=None,
                    group=None, stream=None):
    """One decode step of this rank's shard: the rank's share of m on the GPU,
    the all-reduce of the shares, then the boundary (residual add and RMSNorm)
    on the reduced sum.  dims are the shard's (shard_dims)."""
    from . import moe_decode_layer_partial, moe_tp_boundary
    M, H = x.shape
    m = torch.empty((M, H), dtype=torch.float32, device=x.device)
    moe_decode_layer_partial(dims, shard, x, m, workspace, stream=stream)
    all_reduce_partials(m, group)
    out = torch.empty_like(x) if out is None else out
    residual_out = torch.empty_like(residual) if residual_out is None else residual_out
    moe_tp_boundary(m.view(1, M, H), residual, shard["gain"], out, residual_out, dims.rms_eps, stream=stream)
    return out, residual_out
