"""The no-allocation split-K entry point (collected last on purpose).

splitk_gemm_bf16_noalloc serves callers that cannot allocate device memory
where they run the projection (a plugin's enqueue function, a runtime with
its own fixed pool): it keeps its partial sums in the library's static device
scratch.  Its results must equal those of splitk_gemm_bf16 with a caller
workspace, within the tolerance the split-K parity tests use, on two calls in
a row (the second call reuses the scratch the first one left behind)."""

import numpy as np
import pytest
import torch

import moe_decode_layer_bf16_gb300 as m
from moe_decode_layer_bf16_gb300 import synth
from tests.fixtures_moe import to_np
from oracle import moe_oracle as orc

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,N,K,fp32,split", [(4, 7168, 14336, False, 0), (16, 7168, 14336, False, 0),
                                               (8, 256, 7168, True, 0), (4, 7168, 14336, False, 7)])
def test_noalloc_matches_workspace_entry_point(M, N, K, fp32, split):
    dt = torch.float32 if fp32 else torch.bfloat16
    ws = torch.zeros(m.splitk_gemm_workspace_size(M, N, K, split), dtype=torch.uint8, device="cuda")
    for call in range(2):
        a, w = synth.make_projection(M, N, K, seed=70 + call, device="cuda")
        ref = torch.empty((M, N), dtype=dt, device="cuda")
        got = torch.empty((M, N), dtype=dt, device="cuda")
        m.splitk_gemm_bf16(a, w, ref, ws, alpha=0.75, split_k=split)
        m.splitk_gemm_bf16_noalloc(a, w, got, alpha=0.75, split_k=split)
        torch.cuda.synchronize()
        assert orc.max_abs_rel(to_np(got), to_np(ref)) <= 1e-2
        # same kernel, same split and reduction order: identical bits
        assert torch.equal(got, ref)


def test_noalloc_clears_counters_an_earlier_call_left_set():
    # The whole scratch is filled with 0xff first, as if an earlier call had
    # stopped part-way with every tile counter set.  A call that did not clear
    # all of its counters would leave tiles unfinished (their output stays
    # NaN) or sum the wrong partials.  The shape is the one with the most
    # split tiles whose partial sums fit the scratch: 1984 tiles of 64 rows at
    # 8 tokens, each cut into two segments.
    M, N, K = 8, 64 * 1984, 256
    a, w = synth.make_projection(M, N, K, seed=90, device="cuda")
    ws = torch.zeros(m.splitk_gemm_workspace_size(M, N, K, 2), dtype=torch.uint8, device="cuda")
    ref = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    m.splitk_gemm_bf16(a, w, ref, ws, split_k=2)
    for _ in range(2):
        m.moe_debug_fill_noalloc_scratch(0xFF)
        got = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        m.splitk_gemm_bf16_noalloc(a, w, got, split_k=2)
        torch.cuda.synchronize()
        assert torch.equal(got, ref)


def test_noalloc_rejects_beyond_scratch_limit():
    # 256 tokens of a vocabulary-sized projection need more partial sums than
    # the static scratch holds: refused before anything runs
    a = torch.zeros((256, 1024), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((131072, 1024), dtype=torch.bfloat16, device="cuda")
    c = torch.empty((256, 131072), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(m.MoeError) as e:
        m.splitk_gemm_bf16_noalloc(a, w, c)
    assert e.value.status == m.MOE_ERR_SCRATCH_LIMIT
