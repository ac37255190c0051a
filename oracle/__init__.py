"""CPU oracle of the MoGE layer forward -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA path
(``sparse_router_gemm_global_b300``) and neither imports the other; both
consume the seeded inputs of the ``synth`` package.

The arithmetic lives in ``moge_oracle.c`` (plain C, double accumulation); this
file only marshals numpy arrays and chains the steps in the order the pages
give them (Pangu Pro MoE explainer, section 1): router scores -> global
softmax over all N experts -> top-K' inside each of the M groups -> gates ->
permutation -> expert SwiGLU FFN -> weighted combine, plus the imbalance
score.  Every function below is pinned by a ``-m "not gpu"`` test (see
``tests/test_oracle_*.py``); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moge_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libmoge_oracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile libmoge_oracle.so next to its source (gcc -O2, OpenMP)."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _get():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, vp, c_int = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
            lib.oracle_num_threads.restype = c_int
            lib.oracle_set_num_threads.argtypes = [c_int]
            lib.oracle_router_logits.argtypes = [i64, i64, i64, c_int, vp, vp, vp, vp]
            lib.oracle_softmax.argtypes = [i64, i64, vp, vp]
            lib.oracle_select_grouped.argtypes = [i64, i64, i64, i64, vp, vp]
            lib.oracle_select_global.argtypes = [i64, i64, i64, vp, vp]
            lib.oracle_gates.argtypes = [i64, i64, i64, vp, vp, vp, vp]
            lib.oracle_permute.argtypes = [i64, i64, i64, vp, vp, vp, vp, vp]
            lib.oracle_imbalance.argtypes = [i64, i64, i64, vp, vp]
            lib.oracle_imbalance.restype = ctypes.c_double
            lib.oracle_expert_ffn_pairs.argtypes = [i64, vp, vp, i64, i64, c_int, vp, vp, vp, vp, vp]
            lib.oracle_combine_tokens.argtypes = [i64, vp, i64, vp, vp, i64, i64, c_int, vp, vp, vp,
                                                  vp, vp]
            lib.oracle_combine_rows.argtypes = [i64, i64, i64, c_int, vp, vp, vp, vp]
            _lib = lib
    return _lib


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _dt(a) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"oracle takes fp32 or raw-bf16 (uint16) arrays, got {a.dtype}")


def num_threads() -> int:
    return _get().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _get().oracle_set_num_threads(int(n))


def router_logits(x, w_r, bias=None) -> np.ndarray:
    """fp32(x . W_r^T + b) with double accumulation; x [T,d], W_r [N,d]."""
    dt = _dt(x)
    assert _dt(w_r) == dt
    x, w_r = np.ascontiguousarray(x), np.ascontiguousarray(w_r)
    T, d = x.shape
    N = w_r.shape[0]
    out = np.empty((T, N), dtype=np.float32)
    b = None if bias is None else _c(bias, np.float32)
    _get().oracle_router_logits(T, d, N, dt, x.ctypes.data, w_r.ctypes.data,
                                None if b is None else b.ctypes.data, out.ctypes.data)
    return out


def softmax(logits) -> np.ndarray:
    """Global softmax over all experts, float64 [T,N]."""
    l = _c(logits, np.float32)
    T, N = l.shape
    p = np.empty((T, N), dtype=np.float64)
    _get().oracle_softmax(T, N, l.ctypes.data, p.ctypes.data)
    return p


def select_grouped(logits, M: int, kpg: int) -> np.ndarray:
    """idx [T, M*K'] int32: top-K' of every group, group-major slots."""
    l = _c(logits, np.float32)
    T, N = l.shape
    if N % M or not (1 <= kpg <= N // M):
        raise ValueError("need N % M == 0 and 1 <= K' <= N/M")
    idx = np.empty((T, M * kpg), dtype=np.int32)
    _get().oracle_select_grouped(T, N, M, kpg, l.ctypes.data, idx.ctypes.data)
    return idx


def select_global(logits, K: int) -> np.ndarray:
    """idx [T, K] int32: plain top-K over all experts, rank order."""
    l = _c(logits, np.float32)
    T, N = l.shape
    if not (1 <= K <= N):
        raise ValueError("need 1 <= K <= N")
    idx = np.empty((T, K), dtype=np.int32)
    _get().oracle_select_global(T, N, K, l.ctypes.data, idx.ctypes.data)
    return idx


def gates(idx, p):
    """(gate fp32, gate float64) [T,K]: softmax probability of each chosen expert."""
    idx = _c(idx, np.int32)
    p = _c(p, np.float64)
    T, K = idx.shape
    N = p.shape[1]
    g32 = np.empty((T, K), dtype=np.float32)
    g64 = np.empty((T, K), dtype=np.float64)
    _get().oracle_gates(T, N, K, idx.ctypes.data, p.ctypes.data, g32.ctypes.data, g64.ctypes.data)
    return g32, g64


def permute(idx, N: int) -> dict:
    """counts [N], offsets [N+1], pair_row [T,K], row_token [P]."""
    idx = _c(idx, np.int32)
    T, K = idx.shape
    if idx.size and (idx.min() < 0 or idx.max() >= N):
        raise ValueError("expert index out of range")
    counts = np.empty(N, dtype=np.int32)
    offsets = np.empty(N + 1, dtype=np.int32)
    pair_row = np.empty((T, K), dtype=np.int32)
    row_token = np.empty(T * K, dtype=np.int32)
    _get().oracle_permute(T, K, N, idx.ctypes.data, counts.ctypes.data, offsets.ctypes.data,
                          pair_row.ctypes.data, row_token.ctypes.data)
    return {"counts": counts, "offsets": offsets, "pair_row": pair_row, "row_token": row_token}


def imbalance(counts, T: int, M: int):
    """(group_load [M] int32, score float64) with score = (max - min) / T."""
    c = _c(counts, np.int32)
    N = c.shape[0]
    loads = np.empty(M, dtype=np.int32)
    s = _get().oracle_imbalance(T, N, M, c.ctypes.data, loads.ctypes.data)
    return loads, s


def expert_ffn_pairs(tokens, experts, x, w_gate, w_up, w_down) -> np.ndarray:
    """o [n, d] float64: SwiGLU FFN of expert experts[i] on token tokens[i]."""
    dt = _dt(x)
    tokens = _c(tokens, np.int32)
    experts = _c(experts, np.int32)
    x, w_gate, w_up, w_down = (np.ascontiguousarray(a) for a in (x, w_gate, w_up, w_down))
    d = x.shape[1]
    I = w_gate.shape[1]
    out = np.empty((tokens.shape[0], d), dtype=np.float64)
    _get().oracle_expert_ffn_pairs(tokens.shape[0], tokens.ctypes.data, experts.ctypes.data, d, I, dt,
                                   x.ctypes.data, w_gate.ctypes.data, w_up.ctypes.data,
                                   w_down.ctypes.data, out.ctypes.data)
    return out


def combine_tokens(tokens, idx, gate64, x, w_gate, w_up, w_down) -> np.ndarray:
    """y [n, d] float64 for the listed tokens: sum_k gate[t,k] * FFN_{idx[t,k]}(x[t])."""
    dt = _dt(x)
    tokens = _c(tokens, np.int32)
    idx = _c(idx, np.int32)
    gate64 = _c(gate64, np.float64)
    x, w_gate, w_up, w_down = (np.ascontiguousarray(a) for a in (x, w_gate, w_up, w_down))
    d = x.shape[1]
    I = w_gate.shape[1]
    K = idx.shape[1]
    y = np.empty((tokens.shape[0], d), dtype=np.float64)
    _get().oracle_combine_tokens(tokens.shape[0], tokens.ctypes.data, K, idx.ctypes.data,
                                 gate64.ctypes.data, d, I, dt, x.ctypes.data, w_gate.ctypes.data,
                                 w_up.ctypes.data, w_down.ctypes.data, y.ctypes.data)
    return y


def shared_experts_tokens(tokens, n_routed: int, n_shared: int, x, w_gate, w_up, w_down) -> np.ndarray:
    """[n, d] float64: sum over the shared experts s = 0..S-1 (weights at index N + s) of their
    SwiGLU FFN on each listed token, weight 1.  The explainer's section 2 gives Pangu Pro MoE 4
    shared experts beside the 64 routed ones and nothing more; the reading taken is that every
    token visits every shared expert and their outputs are added to the routed combine."""
    tokens = _c(tokens, np.int32)
    out = np.zeros((tokens.shape[0], x.shape[1]), dtype=np.float64)
    for s in range(n_shared):
        out += expert_ffn_pairs(tokens, np.full(tokens.shape[0], n_routed + s, dtype=np.int32), x, w_gate, w_up,
                                w_down)
    return out


def values64(a) -> np.ndarray:
    """An fp32 or raw-bf16 (uint16) array as exact float64 values (bf16 bits b are the fp32 with
    bits b << 16)."""
    if a.dtype == np.uint16:
        return (np.ascontiguousarray(a).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if a.dtype == np.float32:
        return a.astype(np.float64)
    raise TypeError(f"oracle takes fp32 or raw-bf16 (uint16) arrays, got {a.dtype}")


def residual_tokens(tokens, residual) -> np.ndarray:
    """[n, d] float64: the residual-stream rows of the listed tokens.  The pages describe no
    residual; the reading taken is the transformer block's: the layer's output is added once per
    token to the residual stream r, y = r + sum_k gate_k FFN_k(x) + sum_s FFN_s(x), unweighted."""
    return values64(residual)[_c(tokens, np.int32)]


def combine_rows(rows, pair_row, gate64) -> np.ndarray:
    """y [T, d] float64 = sum_k gate[t,k] * rows[pair_row[t,k]] (the combine step alone)."""
    dt = _dt(rows)
    rows = np.ascontiguousarray(rows)
    pair_row = _c(pair_row, np.int32)
    gate64 = _c(gate64, np.float64)
    T, K = pair_row.shape
    d = rows.shape[1]
    y = np.empty((T, d), dtype=np.float64)
    _get().oracle_combine_rows(T, K, d, dt, rows.ctypes.data, pair_row.ctypes.data, gate64.ctypes.data,
                               y.ctypes.data)
    return y


def route(logits, M: int, kpg: int, mode: str = "grouped") -> dict:
    """Routing of given fp32 logits: idx, gates, permutation, loads, score."""
    l = _c(logits, np.float32)
    T, N = l.shape
    p = softmax(l)
    idx = select_grouped(l, M, kpg) if mode == "grouped" else select_global(l, M * kpg)
    g32, g64 = gates(idx, p)
    perm = permute(idx, N)
    loads, score = imbalance(perm["counts"], T, M)
    out = {"logits": l, "p": p, "idx": idx, "gate": g32, "gate64": g64,
           "group_load": loads, "score": score}
    out.update(perm)
    return out


def layer_forward(x, w_router, bias, w_gate, w_up, w_down, M: int, kpg: int, tokens=None,
                  logits=None, n_shared: int = 0, residual=None) -> dict:
    """The whole MoGE layer for the listed tokens (all tokens if None).

    Routing is computed for every token (the permutation and the loads need
    all of them); the expert FFN and combine only for ``tokens``.  Passing
    ``logits`` replaces the router projection by those scores (used to
    re-run the FFN under another routing).  With ``n_shared`` > 0 the weight
    arrays hold N + n_shared experts and the shared experts' outputs are added
    (see shared_experts_tokens); with ``residual`` [T, d] its rows are added too
    (see residual_tokens).
    """
    if logits is None:
        logits = router_logits(x, w_router, bias)
    r = route(logits, M, kpg)
    T = x.shape[0]
    if tokens is None:
        tokens = np.arange(T, dtype=np.int32)
    r["tokens"] = np.asarray(tokens, dtype=np.int32)
    r["y"] = combine_tokens(r["tokens"], r["idx"], r["gate64"], x, w_gate, w_up, w_down)
    if n_shared:
        r["y"] = r["y"] + shared_experts_tokens(r["tokens"], w_router.shape[0], n_shared, x, w_gate, w_up, w_down)
    if residual is not None:
        r["y"] = r["y"] + residual_tokens(r["tokens"], residual)
    return r
