"""Host-side checks of the C ABI (no GPU needed, no compute call is made).

The library must load, export every function declared in include/moge.h, size
workspaces, and reject bad arguments synchronously, before any launch.
"""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import sparse_router_gemm_global_b300 as moge
from sparse_router_gemm_global_b300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moge.h")

INVALID, UNSUPPORTED, WORKSPACE = 1, 2, 3


def _arena(nbytes=64 << 20):
    """A real 256-byte-aligned buffer that every pointer argument below points into.  Every call
    here must fail its host-side checks before anything is launched; should a regression let one
    through, its kernels would still find mapped memory, large enough for every configuration
    used here: device memory where a GPU is present, host memory otherwise (without a device no
    kernel can be launched at all)."""
    if torch.cuda.is_available():
        t = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        return t, t.data_ptr()
    a = np.zeros(nbytes + 256, dtype=np.uint8)
    return a, (a.ctypes.data + 255) & ~255


_ARENA_KEEP, BUF = _arena()  # BUF: the arena's base address, kept alive by _ARENA_KEEP


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


def call_layer(c, ws_bytes=1 << 40, ws=BUF, **over):
    lib = binding.load()
    args = dict(x=BUF, w_router=BUF, bias=None, w_gate=BUF, w_up=BUF, w_down=BUF, y=BUF)
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
    assert call_layer(cfg(), x=BUF + 4) == INVALID                 # misaligned
    assert call_layer(cfg(d=60)) == UNSUPPORTED                     # bf16 rows not 16-byte multiples
    c = cfg()
    c.weight_dtype = moge.MOGE_F32                                  # mixed dtypes
    assert call_layer(c) == UNSUPPORTED
    c = cfg()
    c.act_dtype = c.weight_dtype = 7
    assert call_layer(c) == UNSUPPORTED
    assert call_layer(cfg(N=2048, M=8)) == UNSUPPORTED              # beyond the routing kernel's limit
    assert call_layer(cfg(), ws=None) == WORKSPACE
    assert call_layer(cfg(), ws=BUF + 16) == WORKSPACE             # workspace must be 256-byte aligned
    assert call_layer(cfg(), ws_bytes=1024) == WORKSPACE


def test_other_calls_reject_before_launch():
    lib = binding.load()
    c = cfg()
    r = ctypes.byref(c)
    ws, n = BUF, 1 << 40
    assert lib.moge_route(r, 0, None, None, None, None, BUF, BUF, ws, n, None) == INVALID   # no scores
    assert lib.moge_route(r, 2, None, None, None, BUF, BUF, BUF, ws, n, None) == INVALID   # bad mode
    assert lib.moge_route(r, 0, None, None, None, BUF, None, BUF, ws, n, None) == INVALID
    assert lib.moge_route(r, 0, BUF, None, None, None, BUF, BUF, ws, n, None) == INVALID   # x w/o W_r
    assert lib.moge_route(r, 0, None, None, None, BUF, BUF, BUF, ws, 16, None) == WORKSPACE
    assert lib.moge_permute(r, None, None, BUF, BUF, None, None, None, ws, n, None) == INVALID
    assert lib.moge_permute(r, BUF, BUF, BUF, BUF, None, None, BUF, ws, n, None) == INVALID  # gather w/o rows
    assert lib.moge_expert_ffn(r, BUF, None, BUF, BUF, BUF, BUF, ws, n, None) == INVALID
    assert lib.moge_expert_ffn(r, BUF, BUF, BUF, BUF, BUF, BUF, ws, 8, None) == WORKSPACE
    assert lib.moge_combine(r, BUF, BUF, None, BUF, None) == INVALID
    assert lib.moge_combine(r, BUF, BUF, BUF + 8, BUF, None) == INVALID
    assert lib.moge_imbalance_score(r, None, None, BUF, None) == INVALID
    assert lib.moge_imbalance_score(r, BUF, None, None, None) == INVALID
    bad = cfg(kpg=0)
    assert lib.moge_imbalance_score(ctypes.byref(bad), BUF, None, BUF, None) == INVALID
    assert lib.moge_reset_device_status(None, None) == INVALID
    assert lib.moge_query_device_status(None, None) == INVALID


def test_routing_only_config_needs_no_hidden_size():
    c = moge.make_config(16384, 0, 64, 8, 2, 0, "f32")
    assert moge.moge_workspace_bytes(c) > 16384 * 64 * 4
    lib = binding.load()
    # logits-input routing validates without d / I; fails here only on the workspace size
    assert lib.moge_route(ctypes.byref(c), 0, None, None, None, BUF, BUF, BUF, BUF, 64, None) == WORKSPACE


def test_imbalance_study_rejects_bad_arguments():
    lib = binding.load()
    f = lib.moge_imbalance_study
    c = cfg(T=64, N=16, M=4, kpg=1)
    assert f(ctypes.byref(c), 4, 1, None, None, BUF, None, None, None) == INVALID      # loads required
    assert f(ctypes.byref(c), -1, 1, None, BUF, BUF, None, None, None) == INVALID     # batches < 0
    assert f(ctypes.byref(c), 4, 1, None, BUF + 4, BUF, None, None, None) == INVALID  # misaligned
    wide = cfg(T=64, N=512, M=4, kpg=1)
    assert f(ctypes.byref(wide), 4, 1, None, BUF, BUF, None, None, None) == UNSUPPORTED
    bad = cfg(T=64, N=15, M=4, kpg=1)
    assert f(ctypes.byref(bad), 4, 1, None, BUF, BUF, None, None, None) == INVALID
    assert f(None, 4, 1, None, BUF, BUF, None, None, None) == INVALID


def test_shared_layer_workspace_and_argument_checks():
    c = cfg(T=64, N=16, M=4, kpg=1)
    base = moge.moge_workspace_bytes(c)
    assert moge.moge_workspace_bytes_shared(c, 0) == base
    assert moge.moge_workspace_bytes_shared(c, 4) > base
    assert moge.moge_workspace_bytes_shared(c, -1) == 0 and moge.moge_workspace_bytes_shared(c, 65) == 0
    lib = binding.load()
    f = lib.moge_layer_forward_shared
    big = 1 << 40
    assert f(ctypes.byref(c), -1, BUF, BUF, None, BUF, BUF, BUF, BUF, None, BUF, big, None) == INVALID
    assert f(ctypes.byref(c), 65, BUF, BUF, None, BUF, BUF, BUF, BUF, None, BUF, big, None) == INVALID
    wide = cfg(T=64, N=1024, M=4, kpg=1)
    assert f(ctypes.byref(wide), 4, BUF, BUF, None, BUF, BUF, BUF, BUF, None, BUF, big, None) == UNSUPPORTED
    small_ws = moge.moge_workspace_bytes_shared(c, 4) - 256
    assert f(ctypes.byref(c), 4, BUF, BUF, None, BUF, BUF, BUF, BUF, None, BUF, small_ws, None) == WORKSPACE


def test_residual_layer_argument_checks():
    """moge_layer_forward_residual: a residual is required (T > 0) and 16-byte aligned; the rest
    are moge_layer_forward_shared's checks.  Every call fails before anything is launched."""
    c = cfg(T=64, N=16, M=4, kpg=1)
    lib = binding.load()
    f = lib.moge_layer_forward_residual
    big = 1 << 40
    args = lambda res, S=4, ws_bytes=big, cc=c: (ctypes.byref(cc), S, BUF, res, BUF, None, BUF, BUF, BUF,  # noqa
                                                 BUF, None, BUF, ws_bytes, None)
    assert f(*args(None)) == INVALID                     # no residual
    assert f(*args(BUF + 8)) == INVALID                 # misaligned residual
    assert f(*args(BUF, S=-1)) == INVALID
    assert f(*args(BUF, ws_bytes=moge.moge_workspace_bytes_shared(c, 4) - 256)) == WORKSPACE
    wide = cfg(T=64, N=1024, M=4, kpg=1)
    assert f(*args(BUF, cc=wide)) == UNSUPPORTED
    assert f(None, 0, BUF, BUF, BUF, None, BUF, BUF, BUF, BUF, None, BUF, big, None) == INVALID


def test_noalloc_permute_checks_match_workspace_permute():
    """moge_permute_noalloc runs moge_permute's own argument checks (the layer shape when rows are
    copied, the routing shape otherwise) before its scratch-size check; every call here is
    rejected before anything is launched."""
    lib = binding.load()
    n = 1 << 40

    def both(c, x=BUF, x_perm=BUF, row_token=BUF, idx=BUF):
        r = ctypes.byref(c)
        a = lib.moge_permute(r, idx, x, BUF, BUF, None, row_token, x_perm, BUF, n, None)
        b = lib.moge_permute_noalloc(r, idx, x, BUF, BUF, None, row_token, x_perm, None)
        return a, b

    mixed = cfg()
    mixed.weight_dtype = moge.MOGE_F32
    cases = [(mixed, UNSUPPORTED),                        # act dtype != weight dtype, rows copied
             (cfg(I=0), INVALID),                         # I < 1, rows copied
             (cfg(d=60), UNSUPPORTED),                    # bf16 rows not 16-byte multiples
             (cfg(d=1 << 21), UNSUPPORTED),               # d beyond 2^20
             (cfg(N=15), INVALID), (cfg(kpg=5), INVALID), (cfg(N=2048, M=8), UNSUPPORTED)]
    for c, want in cases:
        assert both(c) == (want, want), (c.d, c.I, c.N, want)
    assert both(cfg(), row_token=None) == (INVALID, INVALID)       # x_perm needs row_token
    assert both(cfg(), idx=None) == (INVALID, INVALID)
    assert both(cfg(), x=BUF + 4) == (INVALID, INVALID)            # misaligned
