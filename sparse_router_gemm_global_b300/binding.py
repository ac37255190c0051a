"""ctypes binding of libmoge.so with the C function names (argument marshalling only)."""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libmoge.so"

MOGE_F32, MOGE_BF16 = 0, 1
MOGE_ROUTE_GROUPED, MOGE_ROUTE_GLOBAL_TOPK = 0, 1
_STATUS = {0: "MOGE_OK", 1: "MOGE_ERR_INVALID_ARGUMENT", 2: "MOGE_ERR_UNSUPPORTED",
           3: "MOGE_ERR_WORKSPACE", 4: "MOGE_ERR_CUDA", 5: "MOGE_ERR_TIMEOUT"}

_lock = threading.Lock()
_lib = None


class MoGEError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {_STATUS.get(status, status)} ({moge_status_string(status)})")


class Config(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("d", ctypes.c_int64), ("N", ctypes.c_int64), ("M", ctypes.c_int64),
                ("k_per_group", ctypes.c_int64), ("I", ctypes.c_int64), ("act_dtype", ctypes.c_int32),
                ("weight_dtype", ctypes.c_int32)]

    @property
    def K(self) -> int:
        return self.M * self.k_per_group

    @property
    def P(self) -> int:
        return self.T * self.K


class Aux(ctypes.Structure):
    _fields_ = [("logits", ctypes.c_void_p), ("topk_idx", ctypes.c_void_p), ("topk_gate", ctypes.c_void_p),
                ("counts", ctypes.c_void_p), ("offsets", ctypes.c_void_p), ("group_load", ctypes.c_void_p),
                ("score", ctypes.c_void_p)]


def library_path() -> str:
    return os.path.join(PKG, _LIB_NAME)


def load():
    """Load libmoge.so (raises if it is missing: build it with the package's build step)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise ImportError(f"{path} is missing; run `python -m sparse_router_gemm_global_b300.build`")
        lib = ctypes.CDLL(path)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        cfgp = ctypes.POINTER(Config)
        lib.moge_abi_version.restype = i32
        lib.moge_abi_version.argtypes = []
        lib.moge_status_string.restype = ctypes.c_char_p
        lib.moge_status_string.argtypes = [i32]
        lib.moge_workspace_bytes.restype = sz
        lib.moge_workspace_bytes.argtypes = [cfgp]
        lib.moge_reset_device_status.argtypes = [vp, vp]
        lib.moge_query_device_status.argtypes = [vp, vp]
        lib.moge_route.argtypes = [cfgp, i32, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        lib.moge_permute.argtypes = [cfgp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        lib.moge_expert_ffn.argtypes = [cfgp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        lib.moge_combine.argtypes = [cfgp, vp, vp, vp, vp, vp]
        lib.moge_imbalance_score.argtypes = [cfgp, vp, vp, vp, vp]
        lib.moge_layer_forward.argtypes = [cfgp, vp, vp, vp, vp, vp, vp, vp, ctypes.POINTER(Aux), vp, sz, vp]
        lib.moge_permute_noalloc.argtypes = [cfgp, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.moge_permute_noalloc.restype = i32
        lib.moge_workspace_bytes_shared.restype = sz
        lib.moge_workspace_bytes_shared.argtypes = [cfgp, ctypes.c_int64]
        lib.moge_layer_forward_shared.argtypes = [cfgp, ctypes.c_int64, vp, vp, vp, vp, vp, vp, vp,
                                                  ctypes.POINTER(Aux), vp, sz, vp]
        lib.moge_layer_forward_residual.argtypes = [cfgp, ctypes.c_int64, vp, vp, vp, vp, vp, vp, vp, vp,
                                                    ctypes.POINTER(Aux), vp, sz, vp]
        lib.moge_selftest_bounded_wait.argtypes = [vp, ctypes.c_uint64, vp, vp]
        lib.moge_imbalance_study.argtypes = [cfgp, ctypes.c_int64, ctypes.c_uint64, vp, vp, vp, vp, vp, vp]
        lib.moge_set_stage_events.argtypes = [ctypes.POINTER(ctypes.c_void_p), i32]
        lib.moge_kernel_launch_count.restype = ctypes.c_uint64
        lib.moge_kernel_launch_count.argtypes = []
        for fn in ("moge_selftest_bounded_wait", "moge_layer_forward_shared", "moge_layer_forward_residual",
                   "moge_imbalance_study", "moge_set_stage_events", "moge_reset_device_status",
                   "moge_query_device_status", "moge_route", "moge_permute", "moge_expert_ffn", "moge_combine",
                   "moge_imbalance_score", "moge_layer_forward"):
            getattr(lib, fn).restype = i32
        _lib = lib
        return lib


def _ptr(t):
    """Device pointer of a tensor (None -> NULL); raw ints pass through."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise MoGEError(fn, status)


def make_config(T, d, N, M, k_per_group, I, dtype) -> Config:
    dt = {"f32": MOGE_F32, "bf16": MOGE_BF16, MOGE_F32: MOGE_F32, MOGE_BF16: MOGE_BF16}[dtype]
    return Config(T, d, N, M, k_per_group, I, dt, dt)


def moge_abi_version() -> int:
    return load().moge_abi_version()


def moge_status_string(status: int) -> str:
    return load().moge_status_string(status).decode()


def moge_workspace_bytes(cfg: Config) -> int:
    return load().moge_workspace_bytes(ctypes.byref(cfg))


def moge_workspace_bytes_shared(cfg: Config, n_shared: int) -> int:
    return load().moge_workspace_bytes_shared(ctypes.byref(cfg), int(n_shared))


def alloc_workspace(cfg: Config, device="cuda", n_shared: int = 0):
    """A device workspace of moge_workspace_bytes(cfg) bytes (moge_workspace_bytes_shared with
    n_shared > 0) with its status word cleared."""
    import torch
    n = moge_workspace_bytes_shared(cfg, n_shared) if n_shared else moge_workspace_bytes(cfg)
    if n == 0:
        raise MoGEError("moge_workspace_bytes", 1)
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    ws[:4096].zero_()  # status word + self-resetting router counters
    return ws


def moge_reset_device_status(ws, stream=None) -> None:
    _check("moge_reset_device_status", load().moge_reset_device_status(_ptr(ws), _stream(stream)))


def moge_query_device_status(ws, stream=None) -> int:
    """Returns the status code (0 = ok, 5 = a bounded device wait timed out)."""
    return load().moge_query_device_status(_ptr(ws), _stream(stream))


def moge_route(cfg, mode, x, w_router, bias, logits, topk_idx, topk_gate, ws, stream=None) -> None:
    _check("moge_route", load().moge_route(ctypes.byref(cfg), mode, _ptr(x), _ptr(w_router), _ptr(bias),
                                           _ptr(logits), _ptr(topk_idx), _ptr(topk_gate), _ptr(ws),
                                           ws.numel() if ws is not None and not isinstance(ws, int) else 0,
                                           _stream(stream)))


def moge_permute(cfg, topk_idx, x, counts, offsets, pair_row, row_token, x_perm, ws, stream=None) -> None:
    _check("moge_permute", load().moge_permute(ctypes.byref(cfg), _ptr(topk_idx), _ptr(x), _ptr(counts),
                                               _ptr(offsets), _ptr(pair_row), _ptr(row_token), _ptr(x_perm),
                                               _ptr(ws), ws.numel() if ws is not None else 0, _stream(stream)))


def moge_permute_noalloc(cfg, topk_idx, x, counts, offsets, pair_row, row_token, x_perm, stream=None) -> None:
    """moge_permute for callers that cannot hand over a workspace (scratch is a static device array)."""
    _check("moge_permute_noalloc", load().moge_permute_noalloc(
        ctypes.byref(cfg), _ptr(topk_idx), _ptr(x), _ptr(counts), _ptr(offsets), _ptr(pair_row), _ptr(row_token),
        _ptr(x_perm), _stream(stream)))


def moge_expert_ffn(cfg, x_perm, offsets, w_gate, w_up, w_down, y_perm, ws, stream=None) -> None:
    _check("moge_expert_ffn", load().moge_expert_ffn(ctypes.byref(cfg), _ptr(x_perm), _ptr(offsets),
                                                     _ptr(w_gate), _ptr(w_up), _ptr(w_down), _ptr(y_perm),
                                                     _ptr(ws), ws.numel() if ws is not None else 0,
                                                     _stream(stream)))


def moge_combine(cfg, y_perm, pair_row, topk_gate, y, stream=None) -> None:
    _check("moge_combine", load().moge_combine(ctypes.byref(cfg), _ptr(y_perm), _ptr(pair_row),
                                               _ptr(topk_gate), _ptr(y), _stream(stream)))


def moge_imbalance_score(cfg, counts, group_load, score, stream=None) -> None:
    _check("moge_imbalance_score", load().moge_imbalance_score(ctypes.byref(cfg), _ptr(counts),
                                                               _ptr(group_load), _ptr(score), _stream(stream)))


MOGE_NUM_STAGES = 7
STAGE_NAMES = ("route", "permute", "gather", "gate_up", "down", "combine", "imbalance")


def moge_set_stage_events(events) -> None:
    """events: None, or a list of MOGE_NUM_STAGES+1 entries, each a torch.cuda.Event (created with
    timing on) or None (that boundary is not recorded).  The ctypes array is kept alive by the
    binding while recording is on."""
    global _stage_array
    lib = load()
    if events is None:
        _stage_array = None
        _check("moge_set_stage_events", lib.moge_set_stage_events(None, 0))
        return
    handles = []
    for ev in events:
        if ev is None:
            handles.append(None)
            continue
        if not ev.cuda_event:
            ev.record()  # torch creates the underlying cudaEvent_t lazily, on first record
        handles.append(ev.cuda_event)
    arr = (ctypes.c_void_p * len(handles))(*handles)
    _check("moge_set_stage_events", lib.moge_set_stage_events(arr, len(handles)))
    _stage_array = arr


_stage_array = None


def moge_imbalance_study(cfg, batches, seed, bias, loads_grouped, loads_global, is_grouped=None, is_global=None,
                         stream=None) -> None:
    _check("moge_imbalance_study", load().moge_imbalance_study(
        ctypes.byref(cfg), int(batches), int(seed), _ptr(bias), _ptr(loads_grouped), _ptr(loads_global),
        _ptr(is_grouped), _ptr(is_global), _stream(stream)))


def moge_selftest_bounded_wait(ws, timeout_ns, result, stream=None) -> None:
    _check("moge_selftest_bounded_wait", load().moge_selftest_bounded_wait(_ptr(ws), int(timeout_ns), _ptr(result),
                                                                           _stream(stream)))


def moge_kernel_launch_count() -> int:
    return load().moge_kernel_launch_count()


def moge_layer_forward(cfg, x, w_router, bias, w_gate, w_up, w_down, y, ws, aux: dict | None = None,
                       stream=None) -> None:
    a = Aux(*[_ptr((aux or {}).get(k)) for k, _ in Aux._fields_])
    _check("moge_layer_forward", load().moge_layer_forward(
        ctypes.byref(cfg), _ptr(x), _ptr(w_router), _ptr(bias), _ptr(w_gate), _ptr(w_up), _ptr(w_down), _ptr(y),
        ctypes.byref(a), _ptr(ws), ws.numel() if ws is not None else 0, _stream(stream)))


def moge_layer_forward_residual(cfg, n_shared, x, residual, w_router, bias, w_gate, w_up, w_down, y, ws,
                                aux: dict | None = None, stream=None) -> None:
    a = Aux(*[_ptr((aux or {}).get(k)) for k, _ in Aux._fields_])
    _check("moge_layer_forward_residual", load().moge_layer_forward_residual(
        ctypes.byref(cfg), int(n_shared), _ptr(x), _ptr(residual), _ptr(w_router), _ptr(bias), _ptr(w_gate),
        _ptr(w_up), _ptr(w_down), _ptr(y), ctypes.byref(a), _ptr(ws), ws.numel() if ws is not None else 0,
        _stream(stream)))


def moge_layer_forward_shared(cfg, n_shared, x, w_router, bias, w_gate, w_up, w_down, y, ws,
                              aux: dict | None = None, stream=None) -> None:
    a = Aux(*[_ptr((aux or {}).get(k)) for k, _ in Aux._fields_])
    _check("moge_layer_forward_shared", load().moge_layer_forward_shared(
        ctypes.byref(cfg), int(n_shared), _ptr(x), _ptr(w_router), _ptr(bias), _ptr(w_gate), _ptr(w_up),
        _ptr(w_down), _ptr(y), ctypes.byref(a), _ptr(ws), ws.numel() if ws is not None else 0, _stream(stream)))
