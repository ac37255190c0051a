"""Host-side checks of the C ABI (no GPU needed, no compute call is made).

The library must load, export every function declared in include/moge.h, size
workspaces, and reject bad arguments synchronously, before any launch.
"""
import ctypes
import os
import re

import pytest

import sparse_router_gemm_global_b300 as moge
from sparse_router_gemm_global_b300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moge.h")

INVALID, UNSUPPORTED, WORKSPACE = 1, 2, 3
FAKE = 0x7F0000000000  # a well-aligned address that is never dereferenced: every call below fails first


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moge_\w+)\s*\(", src)))


def test_library_exports_every_declared_function():
    lib = binding.load()
    names = declared_functions()
    assert len(names) >= 11
    for n in names:
        assert hasattr(lib, n), n


def test_abi_version_and_status_strings():
    assert moge.moge_abi_version() == 1
    for s in range(6):
        assert moge.moge_status_string(s)
    assert moge.moge_status_string(99) == "unknown status"


def cfg(T=32, d=64, N=16, M=4, kpg=1, I=32, dtype="bf16"):
    return moge.make_config(T, d, N, M, kpg, I, dtype)


def test_workspace_bytes_grows_and_rejects_bad_configs():
    a = moge.moge_workspace_bytes(cfg(T=32))
    b = moge.moge_workspace_bytes(cfg(T=64))
    assert 0 < a < b and a % 256 == 0
    assert moge.moge_workspace_bytes(cfg(N=15, M=4)) == 0          # N % M != 0
    assert moge.moge_workspace_bytes(cfg(kpg=5)) == 0              # K' > G
    assert moge.moge_workspace_bytes(cfg(kpg=0)) == 0
    assert moge.moge_workspace_bytes(cfg(T=-1)) == 0
    assert moge.moge_workspace_bytes(cfg(T=0)) > 0                 # empty batch is valid
    lib = binding.load()
    assert lib.moge_workspace_bytes(None) == 0


def call_layer(c, ws_bytes=1 << 40, ws=FAKE, **over):
    lib = binding.load()
    args = dict(x=FAKE, w_router=FAKE, bias=None, w_gate=FAKE, w_up=FAKE, w_down=FAKE, y=FAKE)
    args.update(over)
    return lib.moge_layer_forward(ctypes.byref(c) if c is not None else None, args["x"], args["w_router"],
                                  args["bias"], args["w_gate"], args["w_up"], args["w_down"], args["y"], None,
                                  ws, ws_bytes, None)


def test_layer_forward_rejects_before_launch():
    assert call_layer(None) == INVALID
    assert call_layer(cfg(N=15)) == INVALID
    assert call_layer(cfg(kpg=5)) == INVALID
    assert call_layer(cfg(d=0)) == INVALID
    assert call_layer(cfg(), x=None) == INVALID
    assert call_layer(cfg(), w_down=None) == INVALID
    assert call_layer(cfg(), x=FAKE + 4) == INVALID                 # misaligned
    assert call_layer(cfg(d=60)) == UNSUPPORTED                     # bf16 rows not 16-byte multiples
    c = cfg()
    c.weight_dtype = moge.MOGE_F32                                  # mixed dtypes
    assert call_layer(c) == UNSUPPORTED
    c = cfg()
    c.act_dtype = c.weight_dtype = 7
    assert call_layer(c) == UNSUPPORTED
    assert call_layer(cfg(N=2048, M=8)) == UNSUPPORTED              # beyond the routing kernel's limit
    assert call_layer(cfg(), ws=None) == WORKSPACE
    assert call_layer(cfg(), ws=FAKE + 16) == WORKSPACE             # workspace must be 256-byte aligned
    assert call_layer(cfg(), ws_bytes=1024) == WORKSPACE


def test_other_calls_reject_before_launch():
    lib = binding.load()
    c = cfg()
    r = ctypes.byref(c)
    ws, n = FAKE, 1 << 40
    assert lib.moge_route(r, 0, None, None, None, None, FAKE, FAKE, ws, n, None) == INVALID   # no scores
    assert lib.moge_route(r, 2, None, None, None, FAKE, FAKE, FAKE, ws, n, None) == INVALID   # bad mode
    assert lib.moge_route(r, 0, None, None, None, FAKE, None, FAKE, ws, n, None) == INVALID
    assert lib.moge_route(r, 0, FAKE, None, None, None, FAKE, FAKE, ws, n, None) == INVALID   # x w/o W_r
    assert lib.moge_route(r, 0, None, None, None, FAKE, FAKE, FAKE, ws, 16, None) == WORKSPACE
    assert lib.moge_permute(r, None, None, FAKE, FAKE, None, None, None, ws, n, None) == INVALID
    assert lib.moge_permute(r, FAKE, FAKE, FAKE, FAKE, None, None, FAKE, ws, n, None) == INVALID  # gather w/o rows
    assert lib.moge_expert_ffn(r, FAKE, None, FAKE, FAKE, FAKE, FAKE, ws, n, None) == INVALID
    assert lib.moge_expert_ffn(r, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ws, 8, None) == WORKSPACE
    assert lib.moge_combine(r, FAKE, FAKE, None, FAKE, None) == INVALID
    assert lib.moge_combine(r, FAKE, FAKE, FAKE + 8, FAKE, None) == INVALID
    assert lib.moge_imbalance_score(r, None, None, FAKE, None) == INVALID
    assert lib.moge_imbalance_score(r, FAKE, None, None, None) == INVALID
    bad = cfg(kpg=0)
    assert lib.moge_imbalance_score(ctypes.byref(bad), FAKE, None, FAKE, None) == INVALID
    assert lib.moge_reset_device_status(None, None) == INVALID
    assert lib.moge_query_device_status(None, None) == INVALID


def test_routing_only_config_needs_no_hidden_size():
    c = moge.make_config(16384, 0, 64, 8, 2, 0, "f32")
    assert moge.moge_workspace_bytes(c) > 16384 * 64 * 4
    lib = binding.load()
    # logits-input routing validates without d / I; fails here only on the workspace size
    assert lib.moge_route(ctypes.byref(c), 0, None, None, None, FAKE, FAKE, FAKE, FAKE, 64, None) == WORKSPACE


def test_imbalance_study_rejects_bad_arguments():
    lib = binding.load()
    f = lib.moge_imbalance_study
    c = cfg(T=64, N=16, M=4, kpg=1)
    assert f(ctypes.byref(c), 4, 1, None, None, FAKE, None, None, None) == INVALID      # loads required
    assert f(ctypes.byref(c), -1, 1, None, FAKE, FAKE, None, None, None) == INVALID     # batches < 0
    assert f(ctypes.byref(c), 4, 1, None, FAKE + 4, FAKE, None, None, None) == INVALID  # misaligned
    wide = cfg(T=64, N=512, M=4, kpg=1)
    assert f(ctypes.byref(wide), 4, 1, None, FAKE, FAKE, None, None, None) == UNSUPPORTED
    bad = cfg(T=64, N=15, M=4, kpg=1)
    assert f(ctypes.byref(bad), 4, 1, None, FAKE, FAKE, None, None, None) == INVALID
    assert f(None, 4, 1, None, FAKE, FAKE, None, None, None) == INVALID


def test_shared_layer_workspace_and_argument_checks():
    c = cfg(T=64, N=16, M=4, kpg=1)
    base = moge.moge_workspace_bytes(c)
    assert moge.moge_workspace_bytes_shared(c, 0) == base
    assert moge.moge_workspace_bytes_shared(c, 4) > base
    assert moge.moge_workspace_bytes_shared(c, -1) == 0 and moge.moge_workspace_bytes_shared(c, 65) == 0
    lib = binding.load()
    f = lib.moge_layer_forward_shared
    big = 1 << 40
    assert f(ctypes.byref(c), -1, FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, None, FAKE, big, None) == INVALID
    assert f(ctypes.byref(c), 65, FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, None, FAKE, big, None) == INVALID
    wide = cfg(T=64, N=1024, M=4, kpg=1)
    assert f(ctypes.byref(wide), 4, FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, None, FAKE, big, None) == UNSUPPORTED
    small_ws = moge.moge_workspace_bytes_shared(c, 4) - 256
    assert f(ctypes.byref(c), 4, FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, None, FAKE, small_ws, None) == WORKSPACE


def test_residual_layer_argument_checks():
    """moge_layer_forward_residual: a residual is required (T > 0) and 16-byte aligned; the rest
    are moge_layer_forward_shared's checks.  Every call fails before anything is launched."""
    c = cfg(T=64, N=16, M=4, kpg=1)
    lib = binding.load()
    f = lib.moge_layer_forward_residual
    big = 1 << 40
    args = lambda res, S=4, ws_bytes=big, cc=c: (ctypes.byref(cc), S, FAKE, res, FAKE, None, FAKE, FAKE, FAKE,  # noqa
                                                 FAKE, None, FAKE, ws_bytes, None)
    assert f(*args(None)) == INVALID                     # no residual
    assert f(*args(FAKE + 8)) == INVALID                 # misaligned residual
    assert f(*args(FAKE, S=-1)) == INVALID
    assert f(*args(FAKE, ws_bytes=moge.moge_workspace_bytes_shared(c, 4) - 256)) == WORKSPACE
    wide = cfg(T=64, N=1024, M=4, kpg=1)
    assert f(*args(FAKE, cc=wide)) == UNSUPPORTED
    assert f(None, 0, FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, None, FAKE, big, None) == INVALID
