"""The C-ABI library loads without a GPU, exports every declared entry point,
and rejects bad arguments on the host before launching anything."""
import ctypes
import os
import re

import pytest

import __graft_entry__ as entry
from expert_routing_moe_gb300 import _abi as abi

HDR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")


def _declared_symbols():
    names = set()
    for fn in os.listdir(HDR):
        if fn.endswith(".h"):
            text = open(os.path.join(HDR, fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", text))
    return names


@pytest.fixture(scope="module")
def lib():
    entry.build()
    return abi.load()


def test_every_declared_symbol_is_exported(lib):
    declared = _declared_symbols()
    assert {"moe_route", "moe_reroute_sere", "moe_dispatch_capacity", "moe_ffn_grouped", "moe_combine",
            "moe_workspace_size", "moe_status_string"} <= declared
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert abi.status_string(0, False) == "ok"
    assert "invalid" in abi.status_string(-1, False)
    assert "timed out" in abi.status_string(abi.MOE_DEV_TIMEOUT, True)


def test_workspace_sizes(lib):
    # bf16 FFN, batches of up to 64 tokens (the decode kernel): counters +
    # the bf16 SwiGLU activations of the whole batch (padded to 16, 32 or 64
    # tokens) for each of the N experts
    bf = abi.workspace_size(abi.MOE_OP_FFN, 32, 2048, 768, 128, 8, 8, False, abi.MOE_DTYPE_BF16)
    assert 128 * 32 * 768 * 2 < bf <= 128 * 32 * 768 * 2 + 4096
    bf1 = abi.workspace_size(abi.MOE_OP_FFN, 1, 2048, 768, 128, 8, 8, False, abi.MOE_DTYPE_BF16)
    assert 128 * 16 * 768 * 2 < bf1 <= 128 * 16 * 768 * 2 + 4096
    # larger batches: the activations of every dispatch row
    bf = abi.workspace_size(abi.MOE_OP_FFN, 128, 2048, 768, 128, 8, 8, False, abi.MOE_DTYPE_BF16)
    assert 128 * 8 * 768 * 2 < bf <= 128 * 8 * 768 * 2 + 4096
    assert abi.workspace_size(abi.MOE_OP_FFN, 32, 64, 128, 8, 2, 2, False, abi.MOE_DTYPE_F32) == 0
    capped = abi.workspace_size(abi.MOE_OP_DISPATCH, 8192, 2048, 768, 128, 8, 10, True, abi.MOE_DTYPE_BF16)
    assert capped >= 2 * 128 * 8192 * 4
    assert abi.workspace_size(abi.MOE_OP_DISPATCH, 8, 64, 64, 0, 2, 2, False, 0) == 0   # N = 0 is invalid


FAKE = ctypes.c_void_p(1 << 20)  # never dereferenced: every call below fails its host-side checks


@pytest.mark.parametrize("args", [
    # T, H, N, R, k
    (4, 64, 0, 2, 2),      # no experts
    (4, 64, 300, 2, 2),    # N above the limit
    (4, 64, 8, 17, 2),     # R above the limit
    (4, 64, 8, 2, 3),      # k > R
    (4, 64, 8, 9, 2),      # R > N
    (-1, 64, 8, 2, 2),     # negative T
])
def test_route_rejects_bad_sizes(lib, args):
    T, H, N, R, k = args
    rc = lib.moe_route(FAKE, 0, FAKE, T, H, N, R, k, 0, FAKE, FAKE, FAKE, None, None, None)
    assert rc == -1


def test_route_rejects_misaligned_and_unsupported(lib):
    odd = ctypes.c_void_p((1 << 20) + 4)
    assert lib.moe_route(odd, 1, FAKE, 4, 64, 8, 2, 2, 0, FAKE, FAKE, FAKE, None, None, None) == -1
    assert lib.moe_route(FAKE, 1, FAKE, 4, 60, 8, 2, 2, 0, FAKE, FAKE, FAKE, None, None, None) == -2  # H % 8
    assert lib.moe_route(FAKE, 0, FAKE, 4, 64, 8, 2, 2, 1 << 7, FAKE, FAKE, FAKE, None, None, None) == -1  # flag
    assert lib.moe_route(None, 0, None, 4, 64, 8, 2, 2, 0, FAKE, FAKE, FAKE, None, None, None) == -1  # no x


def test_route_dispatch_rejects(lib):
    f = lib.moe_route_dispatch
    B = (FAKE, FAKE, FAKE, FAKE, FAKE)           # counts, offsets, row_token, row_gate, active
    W = (FAKE, 1 << 20)
    args = lambda T=32, H=64, N=8, k=2, flags=0, sp=None, ws=W: (FAKE, 1, FAKE, T, H, N, k, flags, FAKE, FAKE, FAKE,
                                                                    sp, *B, *ws, None, None)
    assert f(*args(T=257)) == -2                                # above the single-launch batch limit
    assert f(*args(flags=abi.MOE_ROUTE_FROM_LOGITS)) == -1      # logits are always computed here
    assert f(*args(k=9)) == -1                                  # k > N
    assert f(*args(H=60)) == -2                                 # H % 8 for bf16
    assert f(*args(ws=(None, 0))) == -4                         # no workspace
    assert f(*args(ws=(ctypes.c_void_p((1 << 20) + 16), 1 << 20))) == -1   # misaligned workspace
    sp = abi._SereParams(3, 0.5, FAKE, None, None, None)        # K' > k
    assert f(*args(sp=ctypes.byref(sp))) == -1
    assert abi.workspace_size(abi.MOE_OP_ROUTE_DISPATCH, 32, 2048, 768, 128, 8, 8, False, 1) == 512


def test_decode_layer_rejects(lib):
    f = lib.moe_decode_layer
    W = (FAKE, 1 << 30)
    args = lambda T=32, H=128, I=128, N=8, k=2, rf=0, ff=0, sp=None, y=FAKE, rws=W, fws=W: (
        FAKE, FAKE, FAKE, FAKE, FAKE, T, H, I, N, k, rf, ff, sp, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, y,
        *rws, *fws, None, None)
    assert f(*args(T=65)) == -2                                 # above the decode batch limit
    assert f(*args(T=0)) == -2                                  # an empty batch has nothing to run
    assert f(*args(H=192)) == -2                                # H % 128
    assert f(*args(I=96)) == -2                                 # I % 128
    assert f(*args(k=9)) == -1                                  # k > N
    assert f(*args(rf=abi.MOE_ROUTE_FROM_LOGITS)) == -1         # logits are always computed here
    assert f(*args(ff=abi.MOE_FFN_FUSE_COMBINE)) == -1          # the combine is implied; only ZERO_Y may be set
    assert f(*args(y=None)) == -1                               # no output
    assert f(*args(y=ctypes.c_void_p((1 << 20) + 8))) == -1    # misaligned y
    assert f(*args(rws=(FAKE, 64))) == -4                       # routing workspace too small
    assert f(*args(fws=(FAKE, 64))) == -4                       # FFN workspace too small
    assert f(*args(fws=(ctypes.c_void_p((1 << 20) + 16), 1 << 30))) == -1   # misaligned FFN workspace
    sp = abi._SereParams(3, 0.5, FAKE, None, None, None)        # K' > k
    assert f(*args(sp=ctypes.byref(sp))) == -1


def test_sere_rejects_bad_params(lib):
    sp = abi._SereParams(0, 0.5, FAKE, None, None, None)          # K' = 0
    assert lib.moe_reroute_sere(FAKE, FAKE, 4, 4, 8, 4, ctypes.byref(sp), None, None) == -1
    sp = abi._SereParams(5, 0.5, FAKE, None, None, None)          # K' > k
    assert lib.moe_reroute_sere(FAKE, FAKE, 4, 4, 8, 4, ctypes.byref(sp), None, None) == -1
    sp = abi._SereParams(1, 0.5, None, None, None, None)          # no similarity matrix
    assert lib.moe_reroute_sere(FAKE, FAKE, 4, 4, 8, 4, ctypes.byref(sp), None, None) == -1
    sp = abi._SereParams(1, 0.5, FAKE, None, None, None)
    assert lib.moe_reroute_sere(FAKE, FAKE, 4, 5000, 8, 4, ctypes.byref(sp), None, None) == -2  # T too large
    # fused with ranking: R must equal k
    assert lib.moe_route(FAKE, 0, FAKE, 4, 64, 8, 4, 2, 0, FAKE, FAKE, FAKE, ctypes.byref(sp), None, None) == -1


def test_dispatch_rejects(lib):
    d = lib.moe_dispatch_capacity
    # capped mode needs ld >= R and R >= k
    assert d(FAKE, FAKE, 2, 4, 8, 2, 4, None, 1.25, None, None, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None, None, None,
             None, FAKE, 1 << 30, None, None) == -1
    # capped mode with T above the limit
    assert d(FAKE, FAKE, 4, 20000, 8, 2, 4, None, 1.25, None, None, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None, None, None,
             None, FAKE, 1 << 30, None, None) == -2
    # workspace too small
    assert d(FAKE, FAKE, 4, 64, 8, 2, 4, None, 1.25, None, None, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None, None, None,
             None, FAKE, 16, None, None) == -4
    # a modality bias needs the visual ratio
    assert d(FAKE, FAKE, 4, 64, 8, 2, 4, None, 1.25, FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None,
             None, None, None, FAKE, 1 << 30, None, None) == -1
    # NaN capacity factor
    assert d(FAKE, FAKE, 4, 64, 8, 2, 4, None, float("nan"), None, None, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None, None,
             None, None, FAKE, 1 << 30, None, None) == -1


def test_ffn_rejects(lib):
    f = lib.moe_ffn_grouped
    # bf16 needs H % 128 == 0 and I % 128 == 0
    assert f(FAKE, 1, FAKE, FAKE, FAKE, 4, 96, 128, 8, 2, FAKE, FAKE, FAKE, FAKE, 1, FAKE, FAKE, 1 << 30, None,
             None) == -2
    assert f(FAKE, 1, FAKE, FAKE, FAKE, 4, 128, 96, 8, 2, FAKE, FAKE, FAKE, FAKE, 1, FAKE, FAKE, 1 << 30, None,
             None) == -2   # I % 128
    # misaligned x and a misaligned workspace
    odd = ctypes.c_void_p((1 << 20) + 8)
    assert f(odd, 1, FAKE, FAKE, FAKE, 4, 128, 128, 8, 2, FAKE, FAKE, FAKE, FAKE, 1, FAKE, None, 0, None,
             None) == -1
    assert f(FAKE, 1, FAKE, FAKE, FAKE, 4, 128, 128, 8, 2, FAKE, FAKE, FAKE, FAKE, 1, FAKE, odd, 1 << 20, None,
             None) == -1
    # unknown dtype and unknown flag
    assert f(FAKE, 7, FAKE, FAKE, FAKE, 4, 128, 128, 8, 2, FAKE, FAKE, FAKE, FAKE, 1, FAKE, FAKE, 1 << 30, None,
             None) == -1
    assert f(FAKE, 1, FAKE, FAKE, FAKE, 4, 128, 128, 8, 2, FAKE, FAKE, FAKE, FAKE, 1 << 5, FAKE, FAKE, 1 << 30,
             None, None) == -1


def test_combine_rejects(lib):
    assert lib.moe_combine(FAKE, FAKE, FAKE, 4, 64, 0, FAKE, None) == -1
    assert lib.moe_combine(FAKE, None, FAKE, 4, 64, 2, FAKE, None) == -1


def test_residual_to_bf16_rejects(lib):
    f = lib.moe_residual_to_bf16
    odd = ctypes.c_void_p((1 << 20) + 4)
    assert f(FAKE, FAKE, 12, None) == -1      # n % 8
    assert f(FAKE, FAKE, -8, None) == -1      # negative n
    assert f(odd, FAKE, 16, None) == -1       # misaligned x
    assert f(FAKE, odd, 16, None) == -1       # misaligned y
    assert f(None, FAKE, 16, None) == -1      # no input
    assert f(None, None, 0, None) == 0        # n = 0: nothing to do


def test_token_weights_rejects(lib):
    f = lib.moe_token_weights
    odd = ctypes.c_void_p((1 << 20) + 8)
    W = (FAKE, 1 << 20)
    assert f(FAKE, 1, 4, 64, FAKE, 1.0, 0.0, FAKE, FAKE, None, *W, None, None) == -1     # eps must be > 0
    assert f(FAKE, 1, 4, 64, FAKE, float("nan"), 1e-6, FAKE, FAKE, None, *W, None, None) == -1
    assert f(FAKE, 1, 4, 60, FAKE, 1.0, 1e-6, FAKE, FAKE, None, *W, None, None) == -2    # H % 8
    assert f(odd, 1, 4, 64, FAKE, 1.0, 1e-6, FAKE, FAKE, None, *W, None, None) == -1     # misaligned x
    assert f(FAKE, 5, 4, 64, FAKE, 1.0, 1e-6, FAKE, FAKE, None, *W, None, None) == -1    # dtype
    assert f(FAKE, 1, 4, 64, None, 1.0, 1e-6, FAKE, FAKE, None, *W, None, None) == -1    # no is_visual
    assert f(FAKE, 1, 4, 64, FAKE, 1.0, 1e-6, FAKE, FAKE, None, FAKE, 0, None, None) == -4   # no workspace
    assert f(None, 1, 0, 64, None, 1.0, 1e-6, None, None, None, None, 0, None, None) == 0    # empty batch
    big = (1 << 24) + 1                                                                       # fixed-point range
    assert f(FAKE, 1, big, 64, FAKE, 1.0, 1e-6, FAKE, FAKE, None, *W, None, None) == -2


def test_similarity_calibrate_rejects(lib):
    f = lib.moe_similarity_calibrate
    assert f(FAKE, 16, FAKE, FAKE, FAKE, 256, 128, 200, FAKE, FAKE, 1 << 30, None, None) == -2   # N > 128
    assert f(FAKE, 16, FAKE, FAKE, FAKE, 192, 128, 8, FAKE, FAKE, 1 << 30, None, None) == -2     # H % 128
    assert f(FAKE, 0, FAKE, FAKE, FAKE, 256, 128, 8, FAKE, FAKE, 1 << 30, None, None) == -1      # no tokens
    assert f(FAKE, 16, FAKE, FAKE, FAKE, 256, 128, 8, None, FAKE, 1 << 30, None, None) == -1     # no output
    assert f(FAKE, 16, FAKE, FAKE, FAKE, 256, 128, 8, FAKE, FAKE, 16, None, None) == -4          # workspace
