"""Tensor parallelism on the host: the weight sharding of
moe_decode_layer_bf16_gb300.tp against the oracle's shards, and the rank
choreography (each rank's share of m, the all-reduce, the boundary) as two
CPU processes over gloo, with the oracle standing in for the GPU kernels
(the kernels themselves are checked rank by rank in tests/test_gpu_tp.py)."""

import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from moe_decode_layer_bf16_gb300 import synth, tp
from moe_decode_layer_bf16_gb300.dims import TINY
from oracle import moe_oracle as orc
from tests.fixtures_moe import oracle_layer, tie_free_tokens, to_np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
DIMS = TINY.with_(inter=512, shared_inter=512)


@pytest.mark.parametrize("G", [2, 4])
def test_shard_weights_match_the_oracle_shards(G):
    lw = synth.make_layer(DIMS, seed=3)
    L = oracle_layer(DIMS, lw)
    sd = tp.shard_dims(DIMS, G)
    assert (sd.inter, sd.shared_inter) == (DIMS.inter // G, DIMS.shared_inter // G)
    for g in range(G):
        sw = tp.shard_weights(DIMS, lw, g, G)
        ref = orc.tp_shard(L, g, G)
        for n in ("w13", "w13_s", "w2", "w2_s", "sw13", "sw13_s", "sw2", "sw2_s"):
            assert sw[n].is_contiguous()
            assert np.array_equal(to_np(sw[n]), getattr(ref, n)), n
        assert sw["router_w"] is lw["router_w"]


def test_shard_rejects_splits_that_cut_a_block():
    with pytest.raises(ValueError):
        tp.shard_dims(TINY, 4)  # 256 / 4 = 64: not a whole 128-block
    with pytest.raises(ValueError):
        tp.shard_weights(DIMS, synth.make_layer(DIMS, seed=1), 2, 2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        lw = synth.make_layer(DIMS, seed=5)  # every rank draws the same layer
        x, res, _ = tie_free_tokens(DIMS, lw, 6, seed=5)
        shard = tp.shard_weights(DIMS, lw, rank, world)
        L = oracle_layer(tp.shard_dims(DIMS, world), shard)
        part = orc.moe_decode_layer(L, to_np(x), to_np(res))
        m = torch.from_numpy(part["m"].astype(np.float32))
        tp.all_reduce_partials(m)
        out, ro = orc.rmsnorm_residual(m.numpy().astype(np.float64), to_np(res), to_np(lw["gain"]), DIMS.rms_eps)
        full = orc.moe_decode_layer(oracle_layer(DIMS, lw), to_np(x), to_np(res))
        q.put((rank, orc.max_abs_rel(out, full["out"]), orc.max_abs_rel(ro, full["residual_out"]),
               bool(np.array_equal(part["ids"], full["ids"]))))
    finally:
        dist.destroy_process_group()


def test_tp_layer_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=5) for _ in range(2))
    for rank, e_out, e_res, same_ids in res:
        # fp32 shares summed in another order than the oracle's float64 m
        assert same_ids and e_out <= 1e-2 and e_res <= 1e-2, res
