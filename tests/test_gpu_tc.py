"""The tensor-core (tcgen05) expert kernel against the CPU oracle, through the
C ABI.  moe_set_expert_path forces the kernel, so that the same shapes the
warp-MMA kernel is tested on run here too; the automatic choice is checked to
pick this kernel where it is meant to run (dense layers from 4 tokens, MoE
layers from 16 tokens).  Same bar as tests/test_gpu_parity.py: routing exact,
weights within 1e-5, bf16 outputs within max-abs-rel 2e-2."""

import numpy as np
import pytest
import torch

import moe_decode_layer_bf16_gb300 as m
from moe_decode_layer_bf16_gb300 import synth
from moe_decode_layer_bf16_gb300.dims import DSV3, DSV3_DENSE, TINY, TINY_DENSE
from oracle import moe_oracle as orc
from tests.fixtures_moe import oracle_layer, tie_free_tokens, to_np
from tests.test_gpu_parity import TOL, VARIANTS, LazyLayer, compare, run_gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture
def tc_path():
    m.moe_set_expert_path(m.MOE_PATH_TCGEN05)
    yield
    m.moe_set_expert_path(m.MOE_PATH_AUTO)


# passes of up to 64 tokens: 150 tokens give the shared expert three passes
# (the last of 22 tokens) and the routed experts about 37 tokens each
@pytest.mark.parametrize("M", [1, 4, 13, 33, 150])
def test_tiny_layer_tc(tc_path, M):
    assert m.moe_decode_layer_plan(TINY, M)[0] == m.MOE_PATH_TCGEN05
    lw = synth.make_layer(TINY, seed=0, device=DEV)
    x, res, _ = tie_free_tokens(TINY, lw, M, seed=M, device=DEV)
    compare(TINY, lw, x, res)


@pytest.mark.parametrize("name", sorted(VARIANTS))
@pytest.mark.parametrize("M", [1, 19, 70])
def test_layer_variants_tc(tc_path, name, M):
    dims, kw, zipf = VARIANTS[name]
    lw = synth.make_layer(dims, seed=7, device=DEV, **kw)
    x, res, _ = tie_free_tokens(dims, lw, M, seed=100 + M, zipf=zipf, device=DEV)
    compare(dims, lw, x, res)


def test_tc_outputs_are_deterministic(tc_path):
    dims = TINY.with_(num_experts=64, top_k=8, hidden=1024)
    lw = synth.make_layer(dims, seed=3, device=DEV)
    x, res, _ = tie_free_tokens(dims, lw, 90, seed=3, device=DEV)
    layer = m.MoeDecodeLayer(dims, lw, max_tokens=90)
    a = run_gpu(dims, lw, x, res, layer)
    b = run_gpu(dims, lw, x, res, layer)
    for key in a:
        assert np.array_equal(a[key], b[key]), key


def test_tc_and_warp_paths_share_a_workspace():
    # the two kernels leave the workspace's counters as they found them: calls
    # alternating between them on one workspace all match the oracle
    lw = synth.make_layer(TINY, seed=5, device=DEV)
    layer = m.MoeDecodeLayer(TINY, lw, max_tokens=40)
    L = oracle_layer(TINY, lw)
    try:
        for i, (path, M) in enumerate([(m.MOE_PATH_TCGEN05, 40), (m.MOE_PATH_WARP_MMA, 7),
                                       (m.MOE_PATH_TCGEN05, 3), (m.MOE_PATH_WARP_MMA, 40)]):
            m.moe_set_expert_path(path)
            x, res, _ = tie_free_tokens(TINY, lw, M, seed=60 + i, device=DEV)
            g = run_gpu(TINY, lw, x, res, layer)
            ref = orc.moe_decode_layer(L, to_np(x), to_np(res))
            assert np.array_equal(g["ids"], ref["ids"])
            assert orc.max_abs_rel(g["out"], ref["out"]) <= TOL
    finally:
        m.moe_set_expert_path(m.MOE_PATH_AUTO)


def test_tc_timeout_is_reported_and_gpu_stays_usable(tc_path):
    lw = synth.make_layer(TINY, seed=1, device=DEV)
    x, res, _ = tie_free_tokens(TINY, lw, 4, seed=1, device=DEV)
    layer = m.MoeDecodeLayer(TINY, lw, max_tokens=4)
    m.moe_debug_set_fault(layer.workspace, 1)
    layer(x, res)
    assert layer.status() == m.MOE_ERR_DEVICE_TIMEOUT
    m.moe_debug_set_fault(layer.workspace, 0)
    g = run_gpu(TINY, lw, x, res, layer)
    ref = orc.moe_decode_layer(oracle_layer(TINY, lw), to_np(x), to_np(res))
    assert orc.max_abs_rel(g["out"], ref["out"]) <= TOL


@pytest.mark.parametrize("M", [1, 5, 33, 100])
def test_dense_layer_tiny_tc(tc_path, M):
    lw = synth.make_layer(TINY_DENSE, seed=11, device=DEV)
    x, res = synth.make_tokens(M, TINY_DENSE.hidden, seed=200 + M, device=DEV)
    g = run_gpu(TINY_DENSE, lw, x, res)
    ref = orc.moe_decode_layer(oracle_layer(TINY_DENSE, lw), to_np(x), to_np(res))
    assert orc.max_abs_rel(g["out"], ref["out"]) <= TOL
    assert orc.max_abs_rel(g["residual_out"], ref["residual_out"]) <= TOL


# a dense layer's w13 items are split over H: four segments of 1-2 k-blocks at
# H = 640 (5 k-blocks), two at H = 256; the w2 items over I_s
@pytest.mark.parametrize("hidden", [256, 640])
@pytest.mark.parametrize("M", [1, 7, 33])
def test_dense_layer_split_segments_tc(tc_path, hidden, M):
    dims = TINY_DENSE.with_(hidden=hidden, shared_inter=2560)
    lw = synth.make_layer(dims, seed=13, device=DEV)
    x, res = synth.make_tokens(M, dims.hidden, seed=210 + M, device=DEV)
    g = run_gpu(dims, lw, x, res)
    ref = orc.moe_decode_layer(oracle_layer(dims, lw), to_np(x), to_np(res))
    assert orc.max_abs_rel(g["out"], ref["out"]) <= TOL
    assert orc.max_abs_rel(g["residual_out"], ref["residual_out"]) <= TOL


# ------------------------------------------------------------ full size, automatic choice

@pytest.fixture(scope="module")
def dsv3():
    lw = synth.make_layer(DSV3, seed=0, device=DEV)
    return lw, LazyLayer(DSV3, lw)


@pytest.mark.parametrize("M", [9, 32, 64, 130])
def test_dense_layer_dsv3_tc(M):
    # DeepSeek-V3's dense MLP: from 4 tokens the automatic choice is the
    # tcgen05 kernel; up to 64 tokens its w2 items are split into K segments
    # (partial rows the boundary adds), at 130 tokens three passes
    assert m.moe_decode_layer_plan(DSV3_DENSE, M) == (m.MOE_PATH_TCGEN05, 3)
    lw = synth.make_layer(DSV3_DENSE, seed=12, device=DEV)
    x, res = synth.make_tokens(M, DSV3_DENSE.hidden, seed=300 + M, device=DEV)
    g = run_gpu(DSV3_DENSE, lw, x, res)
    ref = orc.moe_decode_layer(LazyLayer(DSV3_DENSE, lw), to_np(x), to_np(res))
    assert orc.max_abs_rel(g["out"], ref["out"]) <= TOL
    assert orc.max_abs_rel(g["residual_out"], ref["residual_out"]) <= TOL


@pytest.mark.parametrize("M", [64, 256])
def test_dsv3_layer_tc_auto(dsv3, M):
    # verify batches: the automatic choice is the tcgen05 kernel; every active
    # expert's outputs are compared on a covering set of tokens
    assert m.moe_decode_layer_plan(DSV3, M) == (m.MOE_PATH_TCGEN05, 4)
    lw, L = dsv3
    x, res, _ = tie_free_tokens(DSV3, lw, M, seed=3000 + M, device=DEV)
    compare(DSV3, lw, x, res, L=L, cover=True)


@pytest.mark.parametrize("M", [8, 32])
def test_dsv3_layer_tc_forced(tc_path, dsv3, M):
    lw, L = dsv3
    x, res, _ = tie_free_tokens(DSV3, lw, M, seed=3100 + M, device=DEV)
    compare(DSV3, lw, x, res, L=L, cover=True)


@pytest.mark.parametrize("M", [16, 128])
def test_dsv3_skewed_e8m0_tc(tc_path, M):
    # skewed routing: the popular experts hold many tokens (several passes)
    dims = DSV3.with_(e8m0=True)
    lw = synth.make_layer(dims, seed=4, device=DEV, bias_std=0.5, zipf_s=1.1)
    x, res, _ = tie_free_tokens(dims, lw, M, seed=2000 + M, zipf=True, device=DEV)
    compare(dims, lw, x, res, L=LazyLayer(dims, lw), cover=True)
    del lw
    torch.cuda.empty_cache()
