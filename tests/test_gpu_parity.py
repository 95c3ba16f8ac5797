"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Routing (top-k ids, route order, expert offsets) must match exactly; the
routing weights within 1e-5 relative; bf16 outputs within max-abs-rel 2e-2
(|got - ref| / max(|ref|, rms(ref)), per tensor).  Inputs are seeded and
drawn without near-ties in the routing (tests/fixtures_moe.py).
"""

import numpy as np
import pytest
import torch

import moe_decode_layer_bf16_gb300 as m
from moe_decode_layer_bf16_gb300 import synth
from moe_decode_layer_bf16_gb300.dims import DSV3, TINY
from oracle import moe_oracle as orc
from tests.fixtures_moe import oracle_layer, tie_free_tokens, to_np

pytestmark = pytest.mark.gpu
TOL = 2e-2
DEV = "cuda"


class LazyLayer(orc.Layer):
    """Oracle view of a layer whose expert weights stay on the GPU until the
    oracle asks for one expert (the full DeepSeek-V3-shaped layer is 11 GB)."""

    def __init__(self, dims, lw):
        self._lw = lw
        super().__init__(router_w=to_np(lw["router_w"]), sel_bias=to_np(lw["sel_bias"]), w13=None,
                         w13_s=None, w2=None, w2_s=None, sw13=None, sw13_s=None, sw2=None, sw2_s=None,
                         gain=to_np(lw["gain"]), top_k=dims.top_k, routed_scaling=dims.routed_scaling,
                         swiglu_limit=dims.swiglu_limit, rms_eps=dims.rms_eps, e8m0=dims.e8m0,
                         has_shared=lw["sw13"] is not None)

    def expert(self, e):
        if e not in self._cache:
            self._cache.clear()
            lw = self._lw
            if e < 0:
                w = (to_np(lw["sw13"]), to_np(lw["sw13_s"]), to_np(lw["sw2"]), to_np(lw["sw2_s"]))
            else:
                w = (to_np(lw["w13"][e]), to_np(lw["w13_s"][e]), to_np(lw["w2"][e]), to_np(lw["w2_s"][e]))
            self._cache[e] = (orc.dequant_weight(w[0], w[1]), orc.dequant_weight(w[2], w[3]))
        return self._cache[e]


def run_gpu(dims, lw, x, res, layer=None):
    M, k, E = x.shape[0], dims.top_k, dims.num_experts
    layer = layer or m.MoeDecodeLayer(dims, lw, max_tokens=M)
    ids = torch.full((M, k), -1, dtype=torch.int32, device=DEV)
    tw = torch.zeros((M, k), dtype=torch.float32, device=DEV)
    sr = torch.full((M * k,), -1, dtype=torch.int32, device=DEV)
    off = torch.full((E + 1,), -1, dtype=torch.int32, device=DEV)
    out, ro = layer(x, res, topk_ids=ids, topk_w=tw, sorted_routes=sr, expert_offsets=off)
    torch.cuda.synchronize()
    assert layer.status() == m.MOE_OK
    return dict(out=to_np(out), residual_out=to_np(ro), ids=to_np(ids), w=to_np(tw), sorted=to_np(sr),
                off=to_np(off))


def covering_tokens(ids: np.ndarray) -> list:
    """A set of tokens whose routes reach every expert any token was routed
    to: greedily, the token that adds the most experts not yet covered."""
    todo = set(np.unique(ids).tolist())
    rows = [set(r.tolist()) for r in ids]
    chosen = []
    while todo:
        t = max(range(len(rows)), key=lambda i: (len(rows[i] & todo), -i))
        chosen.append(t)
        todo -= rows[t]
    return sorted(chosen)


def compare(dims, lw, x, res, L=None, tokens=None, cover=False):
    """GPU vs oracle.  tokens: the tokens whose outputs are compared (all by
    default); cover=True picks them so that every active routed expert (and
    the shared expert) is checked element by element, after the GPU's routing
    has been checked against the oracle's for every token."""
    g = run_gpu(dims, lw, x, res)
    L = L or oracle_layer(dims, lw)
    if cover:
        _, _, _, ids, _ = orc.route(to_np(x), L.router_w, L.sel_bias, dims.top_k, dims.routed_scaling)
        assert np.array_equal(g["ids"], ids), "top-k ids differ"
        tokens = covering_tokens(ids)
        assert set(np.unique(ids[tokens]).tolist()) == set(np.unique(ids).tolist())
    ref = orc.moe_decode_layer(L, to_np(x), to_np(res), tokens=tokens)
    assert np.array_equal(g["ids"], ref["ids"]), "top-k ids differ"
    assert np.array_equal(g["sorted"], ref["sorted_routes"]), "route order differs"
    assert np.array_equal(g["off"], ref["offsets"]), "expert offsets differ"
    np.testing.assert_allclose(g["w"], ref["weights"], rtol=1e-5, atol=1e-7)
    t = ref["tokens"]
    e_out = orc.max_abs_rel(g["out"][t], ref["out"])
    e_res = orc.max_abs_rel(g["residual_out"][t], ref["residual_out"])
    assert e_out <= TOL and e_res <= TOL, (e_out, e_res)
    return g, ref, e_out, e_res


# ------------------------------------------------------------ small layers

# 150 tokens: passes of 16 tokens; the others: passes of 8 (33: five passes
# of the shared expert, the last with one token)
@pytest.mark.parametrize("M", [1, 4, 13, 33, 150])
def test_tiny_layer(M):
    lw = synth.make_layer(TINY, seed=0, device=DEV)
    x, res, _ = tie_free_tokens(TINY, lw, M, seed=M, device=DEV)
    compare(TINY, lw, x, res)


VARIANTS = {
    "e8m0_bias": (TINY.with_(e8m0=True), dict(bias_std=0.5), False),
    "zipf_e64_k6": (TINY.with_(num_experts=64, top_k=6, hidden=1024), dict(zipf_s=1.1), True),
    "no_shared": (TINY.with_(shared_inter=0), {}, False),
    "shared_wider": (TINY.with_(inter=128, shared_inter=384), {}, False),
    "all_experts": (TINY.with_(num_experts=16, top_k=16), {}, False),
    "uneven_k_split": (TINY.with_(hidden=640, inter=384, shared_inter=128), {}, False),
    "unclamped": (TINY.with_(swiglu_limit=float("inf")), {}, False),
}


@pytest.mark.parametrize("name", sorted(VARIANTS))
@pytest.mark.parametrize("M", [1, 19])
def test_layer_variants(name, M):
    dims, kw, zipf = VARIANTS[name]
    lw = synth.make_layer(dims, seed=7, device=DEV, **kw)
    x, res, _ = tie_free_tokens(dims, lw, M, seed=100 + M, zipf=zipf, device=DEV)
    compare(dims, lw, x, res)


def test_zero_tokens_is_a_no_op():
    lw = synth.make_layer(TINY, seed=2, device=DEV)
    layer = m.MoeDecodeLayer(TINY, lw, max_tokens=4)
    x = torch.empty((0, TINY.hidden), dtype=torch.bfloat16, device=DEV)
    out = torch.empty_like(x)
    layer(x, x, out, out)
    torch.cuda.synchronize()
    assert layer.status() == m.MOE_OK
    # and the workspace still serves a real call afterwards
    xs, res, _ = tie_free_tokens(TINY, lw, 3, seed=2, device=DEV)
    g = run_gpu(TINY, lw, xs, res, layer)
    ref = orc.moe_decode_layer(oracle_layer(TINY, lw), to_np(xs), to_np(res))
    assert np.array_equal(g["ids"], ref["ids"]) and orc.max_abs_rel(g["out"], ref["out"]) <= TOL


def test_outputs_are_deterministic():
    dims = TINY.with_(num_experts=64, top_k=8, hidden=1024)
    lw = synth.make_layer(dims, seed=3, device=DEV)
    x, res, _ = tie_free_tokens(dims, lw, 40, seed=3, device=DEV)
    layer = m.MoeDecodeLayer(dims, lw, max_tokens=40)
    a = run_gpu(dims, lw, x, res, layer)
    b = run_gpu(dims, lw, x, res, layer)
    for key in a:
        assert np.array_equal(a[key], b[key]), key


def test_workspace_reuse_across_token_counts():
    # one workspace sized for 33 tokens serves calls of 33, 1 and 7 tokens
    lw = synth.make_layer(TINY, seed=5, device=DEV)
    layer = m.MoeDecodeLayer(TINY, lw, max_tokens=33)
    L = oracle_layer(TINY, lw)
    for M in (33, 1, 7):
        x, res, _ = tie_free_tokens(TINY, lw, M, seed=50 + M, device=DEV)
        g = run_gpu(TINY, lw, x, res, layer)
        ref = orc.moe_decode_layer(L, to_np(x), to_np(res))
        assert np.array_equal(g["ids"], ref["ids"])
        assert orc.max_abs_rel(g["out"], ref["out"]) <= TOL


def test_timeout_is_reported_and_gpu_stays_usable():
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


# ------------------------------------------------------------ boundary alone

def test_rmsnorm_residual_with_and_without_finalize():
    M, H, k = 5, 1024, 4
    gen = torch.Generator(device=DEV).manual_seed(11)
    rnd = lambda *s: torch.randn(*s, generator=gen, device=DEV)
    x = rnd(M, H).to(torch.bfloat16)
    res = rnd(M, H).to(torch.bfloat16)
    gain = (1 + 0.1 * rnd(H)).to(torch.bfloat16)
    rows = rnd(M * k, H)
    w = rnd(M, k).abs()
    shared = rnd(M, H)
    out = torch.empty_like(res)
    ro = torch.empty_like(res)
    # x only
    m.rmsnorm_residual(res, gain, out, ro, 1e-6, x=x)
    torch.cuda.synchronize()
    ref_o, ref_r = orc.rmsnorm_residual(to_np(x), to_np(res), to_np(gain), 1e-6)
    assert orc.max_abs_rel(to_np(out), ref_o) <= TOL and np.array_equal(to_np(ro), ref_r)
    # finalize of rows + shared
    m.rmsnorm_residual(res, gain, out, ro, 1e-6, rows=rows, route_w=w, shared=shared)
    torch.cuda.synchronize()
    mm = orc.finalize(to_np(rows).astype(np.float64), to_np(w).astype(np.float64), to_np(shared))
    ref_o, ref_r = orc.rmsnorm_residual(mm, to_np(res), to_np(gain), 1e-6)
    assert orc.max_abs_rel(to_np(out), ref_o) <= TOL
    assert orc.max_abs_rel(to_np(ro), ref_r) <= 1e-2


# ------------------------------------------------------------ split-K GEMM

@pytest.mark.parametrize("M", [1, 2, 4, 8, 16])
def test_splitk_eh_proj(M):
    N, K = 7168, 14336
    a, w = synth.make_projection(M, N, K, seed=M, device=DEV)
    c = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    ws = torch.zeros(m.splitk_gemm_workspace_size(M, N, K), dtype=torch.uint8, device=DEV)
    m.splitk_gemm_bf16(a, w, c, ws)
    torch.cuda.synchronize()
    ref = orc.projection(to_np(a), to_np(w))
    assert orc.max_abs_rel(to_np(c), ref) <= 1e-2
    # fp32 sums rounded once to bf16: at most one bf16 ulp from the float64 result
    got = to_np(c)
    ulp = np.abs(ref) * 2.0 ** -7 + 1e-30
    assert (np.abs(got - ref) <= ulp).mean() > 0.999


# explicit splits: one segment per tile (no partial sums), an uneven split of
# the 112 k-blocks (16 each), and one k-block per segment
@pytest.mark.parametrize("split", [1, 7, 112])
@pytest.mark.parametrize("M", [1, 9])
def test_splitk_eh_proj_explicit_split(M, split):
    N, K = 7168, 14336
    a, w = synth.make_projection(M, N, K, seed=80 + M, device=DEV)
    c = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    ws = torch.zeros(m.splitk_gemm_workspace_size(M, N, K, split), dtype=torch.uint8, device=DEV)
    m.splitk_gemm_bf16(a, w, c, ws, split_k=split)
    torch.cuda.synchronize()
    ref = orc.projection(to_np(a), to_np(w))
    got = to_np(c)
    assert orc.max_abs_rel(got, ref) <= 1e-2
    ulp = np.abs(ref) * 2.0 ** -7 + 1e-30
    assert (np.abs(got - ref) <= ulp).mean() > 0.999
    # the counters are left at zero: the same workspace serves the next call alike
    c2 = torch.empty_like(c)
    m.splitk_gemm_bf16(a, w, c2, ws, split_k=split)
    torch.cuda.synchronize()
    assert torch.equal(c, c2)


@pytest.mark.parametrize("M", [1, 8, 16, 33])
def test_splitk_router_form_fp32(M):
    N, K = 256, 7168
    a, w = synth.make_projection(M, N, K, seed=40 + M, device=DEV)
    c = torch.empty((M, N), dtype=torch.float32, device=DEV)
    ws = torch.zeros(m.splitk_gemm_workspace_size(M, N, K), dtype=torch.uint8, device=DEV)
    m.splitk_gemm_bf16(a, w, c, ws, alpha=0.5)
    torch.cuda.synchronize()
    ref = orc.projection(to_np(a), to_np(w), alpha=0.5, out_fp32=True)
    assert orc.max_abs_rel(to_np(c), ref) <= 1e-4


# edge shapes: a last 64-row tile of 16 rows, a single k-block (K = 128),
# token chunks of 32 with a ragged last chunk (M = 17, 33, 255), a single
# 16-row tile (N = 16), fewer cells than CTAs; bf16 and fp32 outputs
@pytest.mark.parametrize("M,N,K", [(1, 1040, 128), (17, 2064, 384), (33, 512, 1024), (255, 1024, 2048),
                                   (5, 16, 7168), (3, 7168, 256)])
def test_splitk_edge_shapes(M, N, K):
    a, w = synth.make_projection(M, N, K, seed=90 + M, device=DEV)
    c = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    ws = torch.zeros(m.splitk_gemm_workspace_size(M, N, K), dtype=torch.uint8, device=DEV)
    m.splitk_gemm_bf16(a, w, c, ws)
    torch.cuda.synchronize()
    ref = orc.projection(to_np(a), to_np(w))
    assert orc.max_abs_rel(to_np(c), ref) <= 1e-2
    c32 = torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV)
    m.splitk_gemm_bf16(a, w, c32, ws)
    torch.cuda.synchronize()
    ref32 = orc.projection(to_np(a), to_np(w), out_fp32=True)
    assert orc.max_abs_rel(to_np(c32), ref32) <= 1e-4


@pytest.mark.parametrize("M", [1, 8])
def test_splitk_lm_head_vocab_width_sampled(M):
    # the LM-head projection at the DeepSeek-V3 vocabulary width (1.85 GB of
    # bf16 weights): 1024 sampled output columns, the first and last included
    N, K = 129280, 7168
    a, w = synth.make_projection(M, N, K, seed=60 + M, device=DEV)
    c = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    ws = torch.zeros(m.splitk_gemm_workspace_size(M, N, K), dtype=torch.uint8, device=DEV)
    m.splitk_gemm_bf16(a, w, c, ws)
    torch.cuda.synchronize()
    cols = np.unique(np.concatenate([[0, N - 1], np.random.default_rng(M).choice(N, 1022, replace=False)]))
    idx = torch.as_tensor(cols, device=DEV)
    ref = orc.projection(to_np(a), to_np(w.index_select(0, idx)))
    assert orc.max_abs_rel(to_np(c)[:, cols], ref) <= 1e-2
    del w


# ------------------------------------------------------------ full-size layers

@pytest.fixture(scope="module")
def dsv3():
    lw = synth.make_layer(DSV3, seed=0, device=DEV)
    return lw, LazyLayer(DSV3, lw)


@pytest.fixture(scope="module")
def dsv3_skewed():
    dims = DSV3.with_(e8m0=True)
    lw = synth.make_layer(dims, seed=4, device=DEV, bias_std=0.5, zipf_s=1.1)
    return dims, lw, LazyLayer(dims, lw)


# Up to 256 tokens the outputs of a set of tokens that reaches every active
# expert are compared element by element (at 64-256 tokens nearly all 256
# experts are active, and above 128 tokens the expert kernel runs 16-token
# passes); 512 tokens (M * k = 4096 routes, the largest step the workspace
# takes) compares the first and the last token.
@pytest.mark.parametrize("M", [1, 8, 32, 64, 128, 256, 512])
def test_dsv3_layer_sampled(dsv3, M):
    lw, L = dsv3
    x, res, _ = tie_free_tokens(DSV3, lw, M, seed=1000 + M, device=DEV)
    if M <= 256:
        compare(DSV3, lw, x, res, L=L, cover=True)
    else:
        compare(DSV3, lw, x, res, L=L, tokens=sorted({0, M - 1}))


@pytest.mark.parametrize("M", [1, 16, 128])
def test_dsv3_skewed_e8m0_sampled(dsv3_skewed, M):
    dims, lw, L = dsv3_skewed
    x, res, _ = tie_free_tokens(dims, lw, M, seed=2000 + M, zipf=True, device=DEV)
    compare(dims, lw, x, res, L=L, cover=True)


# ------------------------------------------------------------ MTP front

def _mtp_inputs(M, H, V, seed):
    gen = torch.Generator(device=DEV).manual_seed(seed)
    rnd = lambda *s: torch.randn(*s, generator=gen, device=DEV)
    ids = torch.randint(0, V, (M,), generator=gen, device=DEV, dtype=torch.int32)
    embed = rnd(V, H).to(torch.bfloat16)
    hidden = (3 * rnd(M, H)).to(torch.bfloat16)
    enorm = (1 + 0.1 * rnd(H)).to(torch.bfloat16)
    hnorm = (1 + 0.1 * rnd(H)).to(torch.bfloat16)
    return ids, embed, hidden, enorm, hnorm


def _run_mtp(ids, embed, hidden, enorm, hnorm, w):
    M, H = hidden.shape
    out = torch.empty((M, H), dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(m.mtp_eh_front_workspace_size(M, H), dtype=torch.uint8, device=DEV)
    m.moe_workspace_init(ws)
    m.mtp_eh_front(ids, embed, hidden, enorm, hnorm, 1e-6, w, out, ws)
    torch.cuda.synchronize()
    assert m.moe_device_status(ws) == m.MOE_OK
    a = ws[256:256 + M * 2 * H * 2].view(torch.bfloat16).view(M, 2 * H)
    return to_np(a), to_np(out)


@pytest.mark.parametrize("M", [1, 3, 17])
def test_mtp_front_small(M):
    H, V = 512, 64
    ids, embed, hidden, enorm, hnorm = _mtp_inputs(M, H, V, seed=M)
    w = (0.02 * torch.randn(H, 2 * H, generator=torch.Generator(device=DEV).manual_seed(9), device=DEV)).to(
        torch.bfloat16)
    a, out = _run_mtp(ids, embed, hidden, enorm, hnorm, w)
    ra, ry = orc.mtp_front(to_np(ids), to_np(embed), to_np(hidden), to_np(enorm), to_np(hnorm), 1e-6, to_np(w))
    # fp32 sums of squares in another order: at most one bf16 ulp off
    ulp = np.abs(ra) * 2.0 ** -7 + 1e-30
    assert (np.abs(a - ra) <= ulp).all()
    assert orc.max_abs_rel(out, ry) <= 1e-2


@pytest.mark.parametrize("M", [1, 8])
def test_mtp_front_dsv3_sampled(M):
    # DeepSeek-V3 sizes: H = 7168, vocabulary 129280 (1.85 GB embedding),
    # eh_proj [7168, 14336]; the input in full, 512 sampled output columns
    H, V = 7168, 129280
    ids, embed, hidden, enorm, hnorm = _mtp_inputs(M, H, V, seed=70 + M)
    _, w = synth.make_projection(1, H, 2 * H, seed=71, device=DEV)
    a, out = _run_mtp(ids, embed, hidden, enorm, hnorm, w)
    e = to_np(embed.index_select(0, ids.long()))
    ra, _ = orc.mtp_front(np.arange(M), e, to_np(hidden), to_np(enorm), to_np(hnorm), 1e-6, np.zeros((1, 2 * H)))
    ulp = np.abs(ra) * 2.0 ** -7 + 1e-30
    assert (np.abs(a - ra) <= ulp).mean() > 0.999 and orc.max_abs_rel(a, ra) <= 1e-2
    cols = np.unique(np.concatenate([[0, H - 1], np.random.default_rng(M).choice(H, 510, replace=False)]))
    ry = orc.projection(ra, to_np(w.index_select(0, torch.as_tensor(cols, device=DEV))))
    assert orc.max_abs_rel(out[:, cols], ry) <= 1e-2


def test_mtp_front_bad_token_id_is_reported():
    H, V, M = 512, 64, 2
    ids, embed, hidden, enorm, hnorm = _mtp_inputs(M, H, V, seed=3)
    ids[1] = V  # one past the table: a zero embedding half and an error status, no read outside
    w = torch.zeros(H, 2 * H, dtype=torch.bfloat16, device=DEV)
    out = torch.empty((M, H), dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(m.mtp_eh_front_workspace_size(M, H), dtype=torch.uint8, device=DEV)
    m.moe_workspace_init(ws)
    m.mtp_eh_front(ids, embed, hidden, enorm, hnorm, 1e-6, w, out, ws)
    torch.cuda.synchronize()
    assert m.moe_device_status(ws) == m.MOE_ERR_INVALID_ARG
    a = to_np(ws[256:256 + M * 2 * H * 2].view(torch.bfloat16).view(M, 2 * H))
    assert not a[1, :H].any() and a[0, :H].any() and a[1, H:].any()


# ------------------------------------------------------------ dense layers

@pytest.mark.parametrize("M", [1, 5, 33])
def test_dense_layer_tiny(M):
    # num_experts = 0: the MLP in the shared-expert slot, no router
    from moe_decode_layer_bf16_gb300.dims import TINY_DENSE
    lw = synth.make_layer(TINY_DENSE, seed=11, device=DEV)
    x, res = synth.make_tokens(M, TINY_DENSE.hidden, seed=200 + M, device=DEV)
    g = run_gpu(TINY_DENSE, lw, x, res)
    ref = orc.moe_decode_layer(oracle_layer(TINY_DENSE, lw), to_np(x), to_np(res))
    assert g["ids"].shape == (M, 0) and np.array_equal(g["off"], [0])
    assert orc.max_abs_rel(g["out"], ref["out"]) <= TOL
    assert orc.max_abs_rel(g["residual_out"], ref["residual_out"]) <= TOL


@pytest.mark.parametrize("M", [1, 8, 32])
def test_dense_layer_dsv3(M):
    # DeepSeek-V3's dense MLP (intermediate 18432, 396 MB of FP8 weights): the
    # w2 items are single 32-row groups there; every token checked
    from moe_decode_layer_bf16_gb300.dims import DSV3_DENSE
    lw = synth.make_layer(DSV3_DENSE, seed=12, device=DEV)
    x, res = synth.make_tokens(M, DSV3_DENSE.hidden, seed=300 + M, device=DEV)
    g = run_gpu(DSV3_DENSE, lw, x, res)
    ref = orc.moe_decode_layer(LazyLayer(DSV3_DENSE, lw), to_np(x), to_np(res))
    assert orc.max_abs_rel(g["out"], ref["out"]) <= TOL
    assert orc.max_abs_rel(g["residual_out"], ref["residual_out"]) <= TOL
