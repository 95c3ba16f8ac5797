"""Tensor-parallel shards on one GPU: each rank's share of m from
moe_decode_layer_partial on its shard, the shares stacked and reduced by
moe_tp_boundary, against the CPU oracle's whole layer (routing exact, outputs
within max-abs-rel 2e-2).  On one GPU the ranks run one after another and the
all-reduce is the boundary's sum over the stacked shares; nothing waits on
another rank."""

import numpy as np
import pytest
import torch

import moe_decode_layer_bf16_gb300 as m
from moe_decode_layer_bf16_gb300 import synth, tp
from moe_decode_layer_bf16_gb300.dims import DSV3, TINY
from oracle import moe_oracle as orc
from tests.fixtures_moe import oracle_layer, tie_free_tokens, to_np
from tests.test_gpu_parity import TOL, LazyLayer, covering_tokens

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_tp(dims, lw, x, res, G):
    M, H = x.shape
    sd = tp.shard_dims(dims, G)
    parts = torch.empty((G, M, H), dtype=torch.float32, device=DEV)
    ids = []
    for g in range(G):
        shard = tp.shard_weights(dims, lw, g, G)
        ws = torch.empty(m.moe_decode_workspace_size(sd, M), dtype=torch.uint8, device=DEV)
        m.moe_workspace_init(ws)
        i = torch.empty((M, dims.top_k), dtype=torch.int32, device=DEV)
        m.moe_decode_layer_partial(sd, shard, x, parts[g], ws, topk_ids=i)
        torch.cuda.synchronize()
        assert m.moe_device_status(ws) == m.MOE_OK
        ids.append(to_np(i))
    out, ro = torch.empty_like(x), torch.empty_like(res)
    m.moe_tp_boundary(parts, res, lw["gain"], out, ro, dims.rms_eps)
    torch.cuda.synchronize()
    return to_np(out), to_np(ro), ids, parts


@pytest.mark.parametrize("path", [m.MOE_PATH_AUTO, m.MOE_PATH_TCGEN05])
@pytest.mark.parametrize("G", [2, 4])
@pytest.mark.parametrize("M", [1, 19])
def test_tp_shards_tiny(M, G, path):
    dims = TINY.with_(inter=512, shared_inter=512)
    lw = synth.make_layer(dims, seed=21, device=DEV)
    x, res, _ = tie_free_tokens(dims, lw, M, seed=400 + M, device=DEV)
    try:
        m.moe_set_expert_path(path)
        out, ro, ids, parts = run_tp(dims, lw, x, res, G)
        # the whole layer on the same GPU, for the shares' sum
        full = m.MoeDecodeLayer(dims, lw, max_tokens=M)
        o_full, r_full = full(x, res)
        torch.cuda.synchronize()
    finally:
        m.moe_set_expert_path(m.MOE_PATH_AUTO)
    ref = orc.moe_decode_layer(oracle_layer(dims, lw), to_np(x), to_np(res))
    for i in ids:
        assert np.array_equal(i, ref["ids"])
    assert orc.max_abs_rel(out, ref["out"]) <= TOL and orc.max_abs_rel(ro, ref["residual_out"]) <= TOL
    # the sum of the shares is the whole layer's m (fp32 summation order apart)
    assert orc.max_abs_rel(to_np(parts.sum(0)), ref["m"]) <= TOL
    assert orc.max_abs_rel(out, to_np(o_full)) <= TOL


def test_tp_boundary_adds_the_shares_in_rank_order():
    # moe_tp_boundary alone: G shares and a residual, against the oracle's
    # boundary over the same shares
    G, M, H = 3, 5, 1024
    gen = torch.Generator(device=DEV).manual_seed(17)
    parts = torch.randn(G, M, H, generator=gen, device=DEV)
    res = torch.randn(M, H, generator=gen, device=DEV).to(torch.bfloat16)
    gain = (1 + 0.1 * torch.randn(H, generator=gen, device=DEV)).to(torch.bfloat16)
    out, ro = torch.empty_like(res), torch.empty_like(res)
    m.moe_tp_boundary(parts, res, gain, out, ro, 1e-6)
    torch.cuda.synchronize()
    o_ref, r_ref = orc.tp_boundary([to_np(p).astype(np.float64) for p in parts], to_np(res), to_np(gain), 1e-6)
    assert orc.max_abs_rel(to_np(out), o_ref) <= TOL and orc.max_abs_rel(to_np(ro), r_ref) <= 1e-2


def test_tp_shards_dsv3_g8():
    # DeepSeek-V3 split 8 ways (I = 256 per rank), 8 tokens, every token compared
    M, G = 8, 8
    lw = synth.make_layer(DSV3, seed=0, device=DEV)
    x, res, _ = tie_free_tokens(DSV3, lw, M, seed=500, device=DEV)
    out, ro, ids, _ = run_tp(DSV3, lw, x, res, G)
    ref = orc.moe_decode_layer(LazyLayer(DSV3, lw), to_np(x), to_np(res))
    for i in ids:
        assert np.array_equal(i, ref["ids"])
    assert orc.max_abs_rel(out, ref["out"]) <= TOL and orc.max_abs_rel(ro, ref["residual_out"]) <= TOL
    del lw
    torch.cuda.empty_cache()
