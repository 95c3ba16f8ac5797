"""The C ABI on the host: the library loads, exports every symbol the header
declares, and rejects bad arguments before touching a GPU.  CPU only."""

import ctypes
import math
import os
import re

import pytest

import moe_decode_layer_bf16_gb300 as m
from moe_decode_layer_bf16_gb300.dims import DSV3, TINY

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_decode.h")


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(m.LIB_PATH):
        from moe_decode_layer_bf16_gb300 import build
        build.build()
    return m.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_three_calls():
    names = declared_functions()
    for n in ("moe_decode_layer", "splitk_gemm_bf16", "rmsnorm_residual"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    for n in declared_functions():
        assert hasattr(L, n), n


def test_status_strings(L):
    assert m.moe_status_str(0) == "ok"
    assert "timed out" in m.moe_status_str(m.MOE_ERR_DEVICE_TIMEOUT)


def test_workspace_size_grows_with_tokens(L):
    sizes = [m.moe_decode_workspace_size(DSV3, t) for t in (1, 8, 32, 256)]
    assert sizes == sorted(sizes) and sizes[0] > 0
    # routed rows (fp32) dominate: at least M*k*H*4 bytes
    assert sizes[-1] >= 256 * 8 * 7168 * 4


@pytest.mark.parametrize("bad,code", [
    (dict(hidden=500), m.MOE_ERR_UNSUPPORTED),
    (dict(inter=200), m.MOE_ERR_UNSUPPORTED),
    (dict(num_experts=600), m.MOE_ERR_UNSUPPORTED),
    (dict(num_experts=20), m.MOE_ERR_UNSUPPORTED),
    (dict(top_k=17), m.MOE_ERR_UNSUPPORTED),
    (dict(top_k=0), m.MOE_ERR_INVALID_ARG),
    (dict(rms_eps=-1.0), m.MOE_ERR_INVALID_ARG),
    (dict(routed_scaling=math.inf), m.MOE_ERR_INVALID_ARG),
])
def test_bad_dims_rejected(L, bad, code):
    with pytest.raises(m.MoeError) as e:
        m.moe_decode_workspace_size(TINY.with_(**bad), 4)
    assert e.value.status == code


def test_dense_dims(L):
    # num_experts = 0 is a dense layer: top_k and inter must be 0, the MLP sits
    # in the shared-expert slot (up to 32768 wide)
    from moe_decode_layer_bf16_gb300.dims import DSV3_DENSE
    assert m.moe_decode_workspace_size(DSV3_DENSE, 32) > 0
    for bad, code in [(dict(top_k=1), m.MOE_ERR_INVALID_ARG), (dict(inter=128), m.MOE_ERR_INVALID_ARG),
                      (dict(shared_inter=0), m.MOE_ERR_INVALID_ARG),
                      (dict(shared_inter=32768 + 128), m.MOE_ERR_UNSUPPORTED)]:
        n = ctypes.c_size_t(0)
        assert L.moe_decode_workspace_size(ctypes.byref(m._dims(DSV3_DENSE.with_(**bad))), 4, ctypes.byref(n)) == code


def test_too_many_tokens_unsupported(L):
    with pytest.raises(m.MoeError) as e:
        m.moe_decode_workspace_size(DSV3, 1024)
    assert e.value.status == m.MOE_ERR_UNSUPPORTED
    # a dense layer (top_k = 0) is bounded by the token count itself
    from moe_decode_layer_bf16_gb300.dims import DSV3_DENSE
    assert m.moe_decode_workspace_size(DSV3_DENSE, 4096) > 0
    with pytest.raises(m.MoeError) as e:
        m.moe_decode_workspace_size(DSV3_DENSE, 4097)
    assert e.value.status == m.MOE_ERR_UNSUPPORTED


def _weights(ptr=0x1000):
    return m._Weights(*[ptr] * len(m._WEIGHT_FIELDS))


def test_layer_rejects_before_launch(L):
    d = m._dims(TINY)
    fake = ctypes.c_void_p(0x10000)
    need = m.moe_decode_workspace_size(TINY, 4)
    # M = 0 is a no-op
    assert L.moe_decode_layer(ctypes.byref(d), ctypes.byref(_weights()), 0, fake, fake, fake, fake,
                              None, None, None, None, fake, need, None) == m.MOE_OK
    # null activation pointer
    assert L.moe_decode_layer(ctypes.byref(d), ctypes.byref(_weights()), 4, None, fake, fake, fake,
                              None, None, None, None, fake, need, None) == m.MOE_ERR_INVALID_ARG
    # misaligned weight
    assert L.moe_decode_layer(ctypes.byref(d), ctypes.byref(_weights(0x1004)), 4, fake, fake, fake, fake,
                              None, None, None, None, fake, need, None) == m.MOE_ERR_INVALID_ARG
    # workspace too small
    assert L.moe_decode_layer(ctypes.byref(d), ctypes.byref(_weights()), 4, fake, fake, fake, fake,
                              None, None, None, None, fake, need - 1, None) == m.MOE_ERR_WORKSPACE_TOO_SMALL
    # more tokens than M*k allows
    assert L.moe_decode_layer(ctypes.byref(d), ctypes.byref(_weights()), 2000, fake, fake, fake, fake,
                              None, None, None, None, fake, need, None) == m.MOE_ERR_UNSUPPORTED


def test_splitk_rejects_before_launch(L):
    fake = ctypes.c_void_p(0x10000)
    call = lambda A, M, N, K, split, ws_bytes: L.splitk_gemm_bf16(A, fake, fake, 0, M, N, K, split, 1.0, fake,
                                                                 ws_bytes, None)
    assert call(fake, 4, 7168, 100, 0, 1 << 30) == m.MOE_ERR_UNSUPPORTED      # K % 128
    assert call(fake, 4, 7000, 14336, 0, 1 << 30) == m.MOE_ERR_UNSUPPORTED    # N % 16
    assert call(fake, 300, 7168, 14336, 0, 1 << 30) == m.MOE_ERR_UNSUPPORTED  # M > 256
    assert call(None, 4, 7168, 14336, 0, 1 << 30) == m.MOE_ERR_INVALID_ARG
    # split_k: negative is invalid, more segments than k-blocks unsupported
    assert call(fake, 4, 7168, 14336, -1, 1 << 30) == m.MOE_ERR_INVALID_ARG
    assert call(fake, 4, 7168, 14336, 113, 1 << 30) == m.MOE_ERR_UNSUPPORTED
    n = ctypes.c_size_t(0)
    assert L.splitk_gemm_workspace_size(4, 7168, 14336, -1, ctypes.byref(n)) == m.MOE_ERR_INVALID_ARG
    assert L.splitk_gemm_workspace_size(4, 7168, 14336, 113, ctypes.byref(n)) == m.MOE_ERR_UNSUPPORTED
    for split in (0, 1, 7, 112):
        need = m.splitk_gemm_workspace_size(4, 7168, 14336, split)
        assert call(fake, 4, 7168, 14336, split, need - 1) == m.MOE_ERR_WORKSPACE_TOO_SMALL
    # an explicit split needs exactly its partial sums: tiles x S x 8 tokens x 64 rows (fp32),
    # none when no tile is split, plus one counter per tile and the two counters of the
    # automatic split's dynamic tail (rounded up to 256 bytes)
    tiles = 7168 // 64
    counters = ((tiles + 2) * 4 + 255) // 256 * 256
    assert m.splitk_gemm_workspace_size(4, 7168, 14336, 1) == counters
    assert m.splitk_gemm_workspace_size(4, 7168, 14336, 7) == counters + tiles * 7 * 8 * 64 * 4
    nz = L.splitk_gemm_bf16_noalloc
    assert nz(fake, fake, fake, 0, 4, 7168, 14336, 113, 1.0, None) == m.MOE_ERR_UNSUPPORTED
    assert nz(fake, fake, fake, 0, 4, 7168, 14336, -2, 1.0, None) == m.MOE_ERR_INVALID_ARG


def test_mtp_front_rejects_before_launch(L):
    fake = ctypes.c_void_p(0x10000)
    call = lambda ids, vocab, eps, M, H, ws_bytes: L.mtp_eh_front(ids, fake, vocab, fake, fake, fake, eps, fake, M, H,
                                                                   fake, fake, ws_bytes, None)
    assert call(fake, 1000, 1e-6, 4, 7000, 1 << 30) == m.MOE_ERR_UNSUPPORTED   # H % 128
    assert call(fake, 1000, 1e-6, 300, 7168, 1 << 30) == m.MOE_ERR_UNSUPPORTED  # M > 256
    assert call(fake, 1000, 1e-6, 0, 7168, 1 << 30) == m.MOE_ERR_INVALID_ARG
    assert call(None, 1000, 1e-6, 4, 7168, 1 << 30) == m.MOE_ERR_INVALID_ARG
    assert call(fake, 0, 1e-6, 4, 7168, 1 << 30) == m.MOE_ERR_INVALID_ARG
    assert call(fake, 1000, -1.0, 4, 7168, 1 << 30) == m.MOE_ERR_INVALID_ARG
    need = m.mtp_eh_front_workspace_size(4, 7168)
    assert need >= 256 + 4 * 2 * 7168 * 2 + m.splitk_gemm_workspace_size(4, 7168, 14336, 0)
    assert call(fake, 1000, 1e-6, 4, 7168, need - 1) == m.MOE_ERR_WORKSPACE_TOO_SMALL


def test_rmsnorm_rejects_before_launch(L):
    fake = ctypes.c_void_p(0x10000)
    assert L.rmsnorm_residual(None, fake, fake, 4, 500, 1e-6, None, None, 0, None, fake, fake, None) == \
        m.MOE_ERR_UNSUPPORTED
    assert L.rmsnorm_residual(None, fake, fake, 4, 512, 1e-6, fake, None, 4, None, fake, fake, None) == \
        m.MOE_ERR_INVALID_ARG
    assert L.rmsnorm_residual(None, None, fake, 4, 512, 1e-6, None, None, 0, None, fake, fake, None) == \
        m.MOE_ERR_INVALID_ARG
    assert L.rmsnorm_residual(None, fake, fake, 0, 512, 1e-6, None, None, 0, None, fake, fake, None) == m.MOE_OK


def test_product_path_has_no_oracle_import():
    pkg = os.path.join(ROOT, "moe_decode_layer_bf16_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"(import\s+oracle|from\s+oracle|oracle[./]|moe_oracle)", src), f


def test_layer_plan_and_path_override(L):
    from moe_decode_layer_bf16_gb300.dims import DSV3_DENSE
    assert m.moe_decode_layer_plan(DSV3, 1) == (m.MOE_PATH_WARP_MMA, 3)
    assert m.moe_decode_layer_plan(DSV3, 8) == (m.MOE_PATH_WARP_MMA, 3)
    assert m.moe_decode_layer_plan(DSV3, 16) == (m.MOE_PATH_TCGEN05, 4)  # + the gather of routed rows
    assert m.moe_decode_layer_plan(DSV3_DENSE, 3) == (m.MOE_PATH_WARP_MMA, 3)
    assert m.moe_decode_layer_plan(DSV3_DENSE, 4) == (m.MOE_PATH_TCGEN05, 3)
    assert m.moe_decode_layer_plan(DSV3, 0) == (m.MOE_PATH_AUTO, 0)
    try:
        m.moe_set_expert_path(m.MOE_PATH_TCGEN05)
        assert m.moe_decode_layer_plan(DSV3, 1) == (m.MOE_PATH_TCGEN05, 4)
        m.moe_set_expert_path(m.MOE_PATH_WARP_MMA)
        assert m.moe_decode_layer_plan(DSV3, 256) == (m.MOE_PATH_WARP_MMA, 3)
    finally:
        m.moe_set_expert_path(m.MOE_PATH_AUTO)
    assert L.moe_set_expert_path(3) == m.MOE_ERR_INVALID_ARG
    p, n = ctypes.c_int(0), ctypes.c_int(0)
    assert L.moe_decode_layer_plan(ctypes.byref(m._dims(DSV3)), 600, ctypes.byref(p), ctypes.byref(n)) == \
        m.MOE_ERR_UNSUPPORTED


def test_workspace_covers_split_dense_rows(L):
    # a dense layer's w2 items may be split into K segments whose partial rows
    # the boundary adds: the workspace holds them and never shrinks as M grows
    from moe_decode_layer_bf16_gb300.dims import DSV3_DENSE
    sizes = [m.moe_decode_workspace_size(DSV3_DENSE, t) for t in range(60, 70)]
    assert sizes == sorted(sizes)
    assert sizes[4] >= 16 * 64 * 7168 * 4  # 64 tokens, up to 16 segments of fp32 rows


def test_tp_entry_points_reject_before_launch(L):
    fake = ctypes.c_void_p(0x10000)
    tb = L.moe_tp_boundary
    assert tb(fake, 0, fake, fake, 4, 512, 1e-6, fake, fake, None) == m.MOE_ERR_INVALID_ARG   # G = 0
    assert tb(fake, 2, fake, fake, 4, 500, 1e-6, fake, fake, None) == m.MOE_ERR_UNSUPPORTED   # H % 128
    assert tb(None, 2, fake, fake, 4, 512, 1e-6, fake, fake, None) == m.MOE_ERR_INVALID_ARG
    assert tb(fake, 2, fake, fake, 0, 512, 1e-6, fake, fake, None) == m.MOE_OK                # M = 0
    d = m._dims(TINY)
    need = m.moe_decode_workspace_size(TINY, 4)
    w = m._Weights(*[0x10000] * len(m._WEIGHT_FIELDS))
    part = L.moe_decode_layer_partial
    # no m_out: invalid; M = 0: a no-op whatever the pointers
    assert part(ctypes.byref(d), ctypes.byref(w), 4, fake, None, None, None, None, None, fake, need, None) == \
        m.MOE_ERR_INVALID_ARG
    assert part(ctypes.byref(d), ctypes.byref(w), 0, None, None, None, None, None, None, None, 0, None) == m.MOE_OK
    # a rank's shard needs no norm gain, but its workspace must fit
    w.norm_gain = None
    assert part(ctypes.byref(d), ctypes.byref(w), 4, fake, fake, None, None, None, None, fake, need - 1, None) == \
        m.MOE_ERR_WORKSPACE_TOO_SMALL
