"""Pins of the CPU oracle against things other than itself: the E4M3 format as
torch implements it, brute-force top-k, sort and sum invariants, library
routines for special cases, and exact integer arithmetic.  CPU only."""

import itertools
import math

import numpy as np
import pytest
import torch

from moe_decode_layer_bf16_gb300 import synth
from moe_decode_layer_bf16_gb300.dims import TINY
from oracle import moe_oracle as orc
from tests.fixtures_moe import oracle_layer, tie_free_tokens, to_np, min_gap


# ---------------------------------------------------------------- FP8 codec

def test_e4m3_decode_matches_torch_for_all_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = orc.e4m3_decode(np.arange(256))
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()
    # landmarks of the format: max 448, min normal 2^-6, min subnormal 2^-9, one NaN per sign
    assert got[0x7E] == 448.0 and got[0x08] == 2.0 ** -6 and got[0x01] == 2.0 ** -9
    assert np.isnan(got[0x7F]) and np.isnan(got[0xFF]) and np.isnan(got).sum() == 2


def test_e4m3_encode_roundtrip_every_finite_code():
    finite = [c for c in range(256) if c not in (0x7F, 0xFF)]
    vals = orc.e4m3_decode(np.array(finite)).astype(np.float32)
    vals[np.array(finite) == 0x80] = np.float32(-0.0)
    assert (orc.e4m3_encode(vals) == np.array(finite, np.uint8)).all()


def test_e4m3_encode_midpoints_round_to_even_and_saturate():
    pos = orc.e4m3_decode(np.arange(127))
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    exact = mids.astype(np.float64) == (pos[:-1] + pos[1:]) / 2
    got = orc.e4m3_encode(mids[exact])
    lo = np.arange(126)[exact]
    want = np.where(lo % 2 == 0, lo, lo + 1)
    assert (got == want).all()
    assert (orc.e4m3_encode(np.float32([449, 464, 500, 1e30])) == 0x7E).all()
    assert (orc.e4m3_encode(np.float32([-449, -1e30])) == 0xFE).all()


def test_e4m3_encode_matches_torch_on_random_values():
    rng = np.random.default_rng(1)
    v = (rng.standard_normal(200_000) * np.exp(rng.uniform(-12, 6, 200_000))).astype(np.float32)
    v = np.clip(v, -448, 448)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = orc.e4m3_encode(v)
    # torch keeps the sign of zero as well
    assert (got == ref).all()


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(2)
    v = (rng.standard_normal(100_000) * 10.0 ** rng.uniform(-5, 5, 100_000)).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    assert (orc.bf16_round(v.astype(np.float64)) == ref).all()


# -------------------------------------------------------------- quantisation

@pytest.mark.parametrize("e8m0", [False, True])
def test_quantize_act_scale_and_error_bound(e8m0):
    rng = np.random.default_rng(3)
    v = (rng.standard_normal((5, 512)) * 3).astype(np.float32)
    v[2, 128:256] = 0.0
    q, s = orc.quantize_act(v, e8m0)
    amax = np.abs(v.reshape(5, 4, 128)).max(axis=2)
    if e8m0:
        nz = amax > 0
        assert (np.log2(s[nz]) == np.round(np.log2(s[nz]))).all()
        assert (s[nz] >= amax[nz] / 448).all() and (s[nz] < 2 * amax[nz] / 448).all()
    else:
        nz = amax > 0
        assert np.array_equal(s[nz], (amax / np.float32(448))[nz])
    assert s[2, 1] == 1.0 and (q[2, 128:256] == 0).all()
    back = orc.dequant_act(q, s)
    # E4M3 keeps 3 mantissa bits: relative error <= 2^-4 above the subnormal range
    big = np.abs(v) > 2.0 ** -6 * s.repeat(128, axis=1)
    rel = np.abs(back - v)[big] / np.abs(v)[big]
    assert rel.max() <= 2.0 ** -4 + 1e-12
    if not e8m0:
        # the group's largest element lands on the largest code
        g = np.abs(v.reshape(5, 4, 128))
        idx = g.argmax(axis=2)
        qq = q.reshape(5, 4, 128)
        top = np.take_along_axis(qq, idx[:, :, None], axis=2)[:, :, 0] & 0x7F
        assert (top[nz] == 0x7E).all()


def test_dequant_weight_block_indexing():
    # codes all 1.0; block sums must equal 128*128*scale of that block.  A
    # transposed scale grid would fail (the grid is 3 x 2, not square).
    codes = np.full((384, 256), 0x38, np.uint8)
    scales = np.arange(1, 7, dtype=np.float32).reshape(3, 2)
    w = orc.dequant_weight(codes, scales)
    sums = w.reshape(3, 128, 2, 128).sum(axis=(1, 3))
    assert np.array_equal(sums, 128 * 128 * scales.astype(np.float64))


# ---------------------------------------------------------------- routing

def test_topk_brute_force_all_subsets():
    rng = np.random.default_rng(4)
    E, k = 16, 4
    for trial in range(20):
        sel = rng.standard_normal((1, E)).astype(np.float32)
        ids = orc.topk_select(sel, k)[0]
        best = max(itertools.combinations(range(E), k), key=lambda c: sum(float(sel[0, e]) for e in c))
        assert set(ids.tolist()) == set(best)
        vals = sel[0, ids]
        assert (np.diff(vals) < 0).all()  # slots in descending selection order
        unsel = np.setdiff1d(np.arange(E), ids)
        assert vals.min() >= sel[0, unsel].max()


def test_topk_tie_goes_to_lower_id():
    sel = np.array([[0.5, 0.9, 0.5, 0.9, 0.1]], np.float32)
    assert orc.topk_select(sel, 3)[0].tolist() == [1, 3, 0]


def test_routing_weight_invariants():
    rng = np.random.default_rng(5)
    logits = rng.standard_normal((7, 16)).astype(np.float32)
    scores = orc.sigmoid_scores(logits)
    bias = rng.standard_normal(16).astype(np.float32) * 0.5
    ids = orc.topk_select(orc.selection_values(scores, bias), 4)
    w = orc.routing_weights(scores, ids, 2.5)
    assert np.allclose(w.sum(axis=1), 2.5, atol=1e-12)
    w1 = orc.routing_weights(scores, ids, 1.0)
    assert np.allclose(w1.sum(axis=1), 1.0, atol=1e-12)
    # weights follow the unbiased scores of the chosen experts
    s = np.take_along_axis(scores.astype(np.float64), ids.astype(np.int64), axis=1)
    assert np.allclose(w1 * s.sum(axis=1, keepdims=True), s)


def test_sigmoid_matches_torch():
    l = np.linspace(-20, 20, 4001).astype(np.float32)
    ref = torch.sigmoid(torch.from_numpy(l).double()).float().numpy()
    assert np.array_equal(orc.sigmoid_scores(l), ref)


def test_route_order_against_brute_force_sort():
    rng = np.random.default_rng(6)
    for M, E, k in [(1, 16, 4), (5, 16, 4), (9, 8, 8), (33, 64, 6)]:
        ids = np.stack([rng.permutation(E)[:k] for _ in range(M)]).astype(np.int32)
        sr, off = orc.route_order(ids, E)
        flat = ids.reshape(-1)
        want = sorted(range(M * k), key=lambda r: (flat[r], r))
        assert sr.tolist() == want
        assert off.tolist() == [0] + np.cumsum(np.bincount(flat, minlength=E)).tolist()


# ---------------------------------------------------------------- MLP pieces

def test_swiglu_unclamped_is_library_silu_times_up():
    rng = np.random.default_rng(7)
    g = rng.standard_normal(1000) * 6
    u = rng.standard_normal(1000) * 6
    ref = (torch.nn.functional.silu(torch.from_numpy(g)) * torch.from_numpy(u)).numpy()
    assert np.allclose(orc.swiglu_clamped(g, u, math.inf), ref, rtol=1e-14, atol=1e-14)


def test_swiglu_clamp_special_values():
    L = 7.0
    # g above the limit is replaced by L; u is clipped on both sides
    assert orc.swiglu_clamped(np.array([50.0]), np.array([-50.0]), L)[0] == pytest.approx(-L * L / (1 + math.exp(-L)))
    assert orc.swiglu_clamped(np.array([-3.0]), np.array([2.0]), L)[0] == pytest.approx(-3.0 / (1 + math.exp(3.0)) * 2.0)


def test_gemms_exact_on_integer_operands():
    # unit scales and integer-valued codes: the FP8 GEMMs must equal an int64 matmul
    rng = np.random.default_rng(8)
    ints = np.arange(-8, 9)
    int_codes = orc.e4m3_encode(ints.astype(np.float32))
    H, I, n = 256, 128, 3
    xi = rng.integers(0, ints.size, (n, H))
    wi = rng.integers(0, ints.size, (2 * I, H))
    xq = int_codes[xi]
    w13 = int_codes[wi]
    x = orc.dequant_act(xq, np.ones((n, H // 128), np.float32))
    w = orc.dequant_weight(w13, np.ones((2, 2), np.float32))
    exact = ints[xi].astype(np.int64) @ ints[wi].astype(np.int64).T
    assert np.array_equal(x @ w.T, exact.astype(np.float64))


def test_dense_average_when_k_equals_e():
    # k = E and equal logits: every expert gets weight scale / E, so the layer's
    # pre-norm sum is the scaled mean of the experts' outputs plus the shared one.
    dims = TINY.with_(num_experts=4, top_k=4)
    lw = synth.make_layer(dims, seed=3)
    lw["router_w"].zero_()
    L = oracle_layer(dims, lw)
    x, res = synth.make_tokens(2, dims.hidden, seed=3)
    out = orc.moe_decode_layer(L, to_np(x), to_np(res))
    assert np.allclose(out["weights"], dims.routed_scaling / 4)
    assert out["ids"].tolist() == [[0, 1, 2, 3]] * 2
    xq, xs = out["xq"], out["xs"]
    ys = [orc.expert_mlp(xq, xs, *L.expert(e), L.swiglu_limit, L.e8m0)[0] for e in range(4)]
    sh = orc.expert_mlp(xq, xs, *L.expert(-1), L.swiglu_limit, L.e8m0)[0]
    want = dims.routed_scaling * np.mean(ys, axis=0) + sh
    assert np.allclose(out["m"], want, rtol=1e-12, atol=1e-12)


def test_rmsnorm_unit_rms_before_gain():
    rng = np.random.default_rng(9)
    m = rng.standard_normal((6, 512)) * 3
    res = orc.bf16_round(rng.standard_normal((6, 512)))
    out, rb = orc.rmsnorm_residual(m, res, np.ones(512), 1e-6)
    assert np.allclose(np.sqrt((out ** 2).mean(axis=1)), 1.0, atol=3e-3)
    assert np.array_equal(rb, orc.bf16_round(m + res))


def test_projection_matches_torch_matmul():
    a, w = synth.make_projection(4, 256, 512, seed=1)
    got = orc.projection(to_np(a), to_np(w))
    ref = (a.double() @ w.double().T).to(torch.bfloat16).double().numpy()
    # a float64 sum rounded once vs torch's double sum rounded once
    assert np.array_equal(got, ref) or np.abs(got - ref).max() <= np.abs(ref).max() * 2 ** -8


# ---------------------------------------------------------------- whole layer

def test_layer_tiny_invariants():
    dims = TINY
    lw = synth.make_layer(dims, seed=0)
    L = oracle_layer(dims, lw)
    x, res, _ = tie_free_tokens(dims, lw, 4, seed=0)
    out = orc.moe_decode_layer(L, to_np(x), to_np(res))
    M, k = 4, dims.top_k
    assert np.allclose(out["weights"].sum(axis=1), dims.routed_scaling)
    assert sorted(out["sorted_routes"].tolist()) == list(range(M * k))
    assert np.array_equal(out["residual_out"], orc.bf16_round(out["m"] + to_np(res)))
    # a subset of tokens gives the same outputs for those tokens
    sub = orc.moe_decode_layer(L, to_np(x), to_np(res), tokens=[2])
    assert np.array_equal(sub["out"][0], out["out"][2])
    assert min_gap(to_np(x), to_np(lw["router_w"]), None, k).min() >= 1e-4


def test_zipf_router_skews_popularity():
    dims = TINY.with_(num_experts=64, top_k=4)
    lw = synth.make_layer(dims, seed=5, zipf_s=1.1)
    x, _ = synth.make_tokens(256, dims.hidden, seed=5, zipf=True)
    _, _, _, ids, _ = orc.route(to_np(x), to_np(lw["router_w"]), None, dims.top_k, 2.5)
    counts = np.sort(np.bincount(ids.reshape(-1), minlength=64))[::-1]
    # the most popular quarter of experts takes most of the routes
    assert counts[:16].sum() > 0.6 * counts.sum()


def test_expert_mlp_gate_rows_then_up_rows():
    # x = 1 everywhere; gate row i reads a_i from column 0, up row i reads 1.
    # Then h_i = silu(min(a_i, L)) and, with w2 = identity, y ~= h within FP8
    # error.  Swapping the halves (g = 1, u = a) would give silu(1) * a.
    H = I = 128
    a = np.linspace(-6, 12, I).astype(np.float32)
    w13 = np.zeros((2 * I, H), np.uint8)
    w13[:I, 0] = orc.e4m3_encode(a)
    w13[I:, 0] = orc.e4m3_encode(np.float32([1.0]))[0]
    a_q = orc.e4m3_decode(w13[:I, 0])
    w2 = np.zeros((H, I), np.uint8)
    w2[np.arange(H), np.arange(I)] = orc.e4m3_encode(np.float32([1.0]))[0]
    xq = np.full((1, H), orc.e4m3_encode(np.float32([1.0]))[0], np.uint8)
    one = np.ones((1, 1), np.float32)
    y, h32, _, _ = orc.expert_mlp(xq, one, orc.dequant_weight(w13, np.ones((2, 1), np.float32)),
                                  orc.dequant_weight(w2, one), 7.0, False)
    want = np.minimum(a_q, 7.0) / (1 + np.exp(-np.minimum(a_q, 7.0)))
    assert np.allclose(h32[0], want, rtol=1e-6)
    assert np.allclose(y[0], want, rtol=2.0 ** -4, atol=1e-3)


def test_shared_expert_term_present_only_when_given():
    # the same layer with and without its shared expert differs by exactly
    # the shared expert's output (pre-norm sum m)
    lw = synth.make_layer(TINY, seed=2)
    x, res = synth.make_tokens(3, TINY.hidden, seed=2)
    with_sh = orc.moe_decode_layer(oracle_layer(TINY, lw), to_np(x), to_np(res))
    L = oracle_layer(TINY, lw)
    L.has_shared = False
    without = orc.moe_decode_layer(L, to_np(x), to_np(res))
    sh = orc.expert_mlp(with_sh["xq"], with_sh["xs"], *L.expert(-1), L.swiglu_limit, L.e8m0)[0]
    assert np.allclose(with_sh["m"] - without["m"], sh, rtol=1e-12, atol=1e-12)
    assert np.abs(sh).max() > 0.1


# ------------------------------------------------------------ MTP front

def _cos(a, b):
    a = np.asarray(a, np.float64).ravel()
    b = np.asarray(b, np.float64).ravel()
    return float(a @ b / np.sqrt((a @ a) * (b @ b)))


def test_mtp_front_halves_order_gather_and_norm():
    # projections that select one half of the concatenated input pin the
    # order (embedding first), the gather and the normalisation by properties:
    # unit RMS with unit gains, the direction of the selected row, and
    # invariance to the row's scale
    rng = np.random.default_rng(5)
    H, V, M = 256, 16, 3
    embed = orc.bf16_round(rng.standard_normal((V, H)))
    hidden = orc.bf16_round(3.0 * rng.standard_normal((M, H)))
    ones = np.ones(H)
    ids = np.array([3, 11, 3])
    eye, zero = np.eye(H), np.zeros((H, H))
    _, ye = orc.mtp_front(ids, embed, hidden, ones, ones, 1e-6, np.concatenate([eye, zero], axis=1))
    _, yh = orc.mtp_front(ids, embed, hidden, ones, ones, 1e-6, np.concatenate([zero, eye], axis=1))
    for t in range(M):
        assert abs(orc.rms(ye[t]) - 1) < 1e-2 and abs(orc.rms(yh[t]) - 1) < 1e-2
        assert _cos(ye[t], embed[ids[t]]) > 0.9999
        assert _cos(yh[t], hidden[t]) > 0.9999
        assert abs(_cos(ye[t], embed[(ids[t] + 1) % V])) < 0.3  # not a neighbouring row
    assert np.array_equal(ye[0], ye[2])  # same token id, same row
    # scale invariance of the normalisation (power-of-two scale: exact in bf16)
    _, ye4 = orc.mtp_front(ids, 4.0 * embed, hidden, ones, ones, 1e-6, np.concatenate([eye, zero], axis=1))
    assert np.array_equal(ye, ye4)
    # gains multiply elementwise after the normalisation: a gain of 2 doubles the half
    _, ye2 = orc.mtp_front(ids, embed, hidden, 2 * ones, ones, 1e-6, np.concatenate([eye, zero], axis=1))
    assert np.array_equal(ye2, 2 * ye)


def test_dense_layer_is_the_moe_layer_without_routed_weight():
    # the dense path (no router, no experts) against the MoE path whose routed
    # contribution is scaled away (routed_scaling = 0): same shared expert, same
    # boundary, so the outputs must agree exactly
    from moe_decode_layer_bf16_gb300 import synth
    from moe_decode_layer_bf16_gb300.dims import TINY
    lw = synth.make_layer(TINY, seed=3)
    x, res = synth.make_tokens(5, TINY.hidden, seed=3)
    L = oracle_layer(TINY.with_(routed_scaling=0.0), lw)
    moe = orc.moe_decode_layer(L, to_np(x), to_np(res))
    dense = orc.Layer(router_w=np.zeros((0, TINY.hidden)), sel_bias=None, w13=None, w13_s=None, w2=None,
                      w2_s=None, sw13=L.sw13, sw13_s=L.sw13_s, sw2=L.sw2, sw2_s=L.sw2_s, gain=L.gain,
                      top_k=0, routed_scaling=0.0, swiglu_limit=L.swiglu_limit, rms_eps=L.rms_eps,
                      e8m0=L.e8m0)
    d = orc.moe_decode_layer(dense, to_np(x), to_np(res))
    assert np.array_equal(d["out"], moe["out"]) and np.array_equal(d["residual_out"], moe["residual_out"])
    assert d["ids"].shape == (5, 0) and np.any(d["out"] != 0)


# ------------------------------------------------------------ finalize

def test_finalize_pairs_each_slot_with_its_own_row():
    # one-hot rows: row r = t*k + j is the unit vector of column r, and slot j
    # of token t carries weight j + 1.  Then m[t, t*k + j] must be j + 1 and
    # every other column of token t zero; pairing slot j with the row of
    # another slot, or another token's rows, moves or changes those values.
    M, k = 3, 4
    H = M * k + 2
    rows = np.eye(M * k, H)
    w = np.tile(np.arange(1, k + 1, dtype=np.float64), (M, 1))
    m = orc.finalize(rows, w, None)
    want = np.zeros((M, H))
    for t in range(M):
        for j in range(k):
            want[t, t * k + j] = j + 1
    assert np.array_equal(m, want)
    # the shared output adds once per token, unweighted
    shared = np.arange(M * H, dtype=np.float64).reshape(M, H)
    assert np.array_equal(orc.finalize(rows, w, shared), want + shared)


def test_routed_part_scales_linearly_with_routed_scaling():
    # the routed scaling multiplies the routed weights only: with the ids
    # unchanged (selection ignores the scaling), m - shared scales by the
    # ratio of the two factors, and the shared expert's output does not
    lw = synth.make_layer(TINY, seed=6)
    x, res, _ = tie_free_tokens(TINY, lw, 3, seed=6)
    a = orc.moe_decode_layer(oracle_layer(TINY.with_(routed_scaling=2.5), lw), to_np(x), to_np(res))
    b = orc.moe_decode_layer(oracle_layer(TINY.with_(routed_scaling=1.0), lw), to_np(x), to_np(res))
    assert np.array_equal(a["ids"], b["ids"])
    assert np.array_equal(a["shared"], b["shared"]) and np.abs(a["shared"]).max() > 0.1
    ra, rb = a["m"] - a["shared"], b["m"] - b["shared"]
    assert np.abs(rb).max() > 0.01
    assert np.allclose(ra, 2.5 * rb, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------ tensor parallelism

@pytest.mark.parametrize("G", [2, 4])
def test_tp_shards_sum_to_the_full_layer(G):
    # each rank keeps I/G of every expert; the ranks' shares of m must add up
    # to the whole layer's m, their h must be slices of the whole layer's h
    # (no quantisation group straddles two ranks), and the boundary over the
    # shares must give the whole layer's outputs
    dims = TINY.with_(inter=512, shared_inter=512)
    lw = synth.make_layer(dims, seed=9)
    L = oracle_layer(dims, lw)
    x, res, _ = tie_free_tokens(dims, lw, 5, seed=9)
    full = orc.moe_decode_layer(L, to_np(x), to_np(res))
    parts = [orc.moe_decode_layer(orc.tp_shard(L, g, G), to_np(x), to_np(res)) for g in range(G)]
    for p in parts:
        assert np.array_equal(p["ids"], full["ids"]) and np.array_equal(p["sorted_routes"], full["sorted_routes"])
    msum = sum(p["m"] for p in parts)
    assert np.allclose(msum, full["m"], rtol=1e-10, atol=1e-12)
    I = dims.inter // G
    for r, h in full["h_rows"].items():
        for g, p in enumerate(parts):
            assert np.allclose(p["h_rows"][r], h[g * I:(g + 1) * I], rtol=1e-6, atol=1e-7)
    out, ro = orc.tp_boundary([p["m"] for p in parts], to_np(res), L.gain, L.rms_eps)
    # the same m up to float64 summation order: equal bf16 outputs, or one bf16 step apart
    assert np.all(np.abs(out - full["out"]) <= np.abs(full["out"]) * 2.0 ** -7)
    assert np.all(np.abs(ro - full["residual_out"]) <= np.abs(full["residual_out"]) * 2.0 ** -7)


def test_tp_shard_with_a_wrong_slice_is_caught():
    # the sum pin catches a shard that takes the up rows from the wrong place
    dims = TINY.with_(inter=512, shared_inter=512)
    lw = synth.make_layer(dims, seed=10)
    L = oracle_layer(dims, lw)
    x, res, _ = tie_free_tokens(dims, lw, 3, seed=10)
    full = orc.moe_decode_layer(L, to_np(x), to_np(res))
    parts = [orc.tp_shard(L, g, 2) for g in range(2)]
    bad = parts[1]
    bad.w13 = bad.w13.copy()
    bad.w13[:, 256:, :] = L.w13[:, 256:512, :]  # rank 1's up rows replaced by gate rows
    ms = [orc.moe_decode_layer(p, to_np(x), to_np(res))["m"] for p in parts]
    assert not np.allclose(ms[0] + ms[1], full["m"], rtol=1e-3, atol=1e-3)
