"""Seeded synthetic inputs shared by the CPU oracle and the CUDA path.

This module only draws numbers (counter-based splitmix64 + Box-Muller, see
``synth.c``); it holds none of the layer's arithmetic.  Every array is
returned as host numpy memory: fp32 arrays as ``float32``, bf16 arrays as raw
``uint16`` bit patterns (use :func:`bf16_to_f32` to read them as values).

Tensor ids (one independent stream each):

====  =====================================================
 id   tensor
====  =====================================================
 1    x            [T, d]        N(0, 1)
 2    W_r          [N, d]        N(0, 1/d)
 3    W_gate       [N, I, d]     N(0, 1/d)
 4    W_up         [N, I, d]     N(0, 1/d)
 5    W_down       [N, d, I]     N(0, 1/I)
 6    rank perm    [N]           Fisher-Yates permutation of 1..N
 7    logit noise  [T, N]        N(0, 1) (routing-only workload)
 8    study scores [B, T, N]     Irwin-Hall(12) ~ N(0, 1), bit-exact by construction
                                 (imbalance Monte-Carlo study; see synth.c)
====  =====================================================
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .workloads import WORKLOADS, Workload, DEFAULT_SEED  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None

TID_X, TID_WR, TID_WGATE, TID_WUP, TID_WDOWN, TID_RANK, TID_LOGIT_NOISE, TID_STUDY = 1, 2, 3, 4, 5, 6, 7, 8
BIAS_SCALE = 1.5


def build(force: bool = False) -> str:
    """Compile libsynth.so next to its source (gcc, OpenMP)."""
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
            u64, i64, dbl = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double
            vp = ctypes.c_void_p
            lib.synth_normal_f32.argtypes = [u64, u64, u64, u64, dbl, vp]
            lib.synth_normal_bf16.argtypes = [u64, u64, u64, u64, dbl, vp]
            lib.synth_f32_to_bf16.argtypes = [vp, u64, vp]
            lib.synth_rank_permutation.argtypes = [u64, u64, i64, vp]
            lib.synth_rank_bias.argtypes = [vp, i64, dbl, vp]
            lib.synth_study_scores.argtypes = [u64, u64, i64, i64, i64, i64, vp]
            lib.synth_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def num_threads() -> int:
    return _get().synth_num_threads()


def normal(seed: int, tensor_id: int, shape, std: float, dtype: str = "f32",
           start: int = 0) -> np.ndarray:
    """Elements [start, start+prod(shape)) of stream ``tensor_id`` as an array."""
    count = int(np.prod(shape)) if len(shape) else 1
    lib = _get()
    if dtype == "f32":
        out = np.empty(shape, dtype=np.float32)
        lib.synth_normal_f32(seed, tensor_id, start, count, float(std), out.ctypes.data)
    elif dtype == "bf16":
        out = np.empty(shape, dtype=np.uint16)
        lib.synth_normal_bf16(seed, tensor_id, start, count, float(std), out.ctypes.data)
    else:
        raise ValueError(dtype)
    return out


def f32_to_bf16(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.uint16)
    _get().synth_f32_to_bf16(a.ctypes.data, a.size, out.ctypes.data)
    return out


def bf16_to_f32(a: np.ndarray) -> np.ndarray:
    """Exact widening of raw bf16 bits to fp32 values."""
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return (a.astype(np.uint32) << 16).view(np.float32)


def rank_permutation(seed: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    _get().synth_rank_permutation(seed, TID_RANK, n, out.ctypes.data)
    return out


def router_bias(seed: int, n: int) -> np.ndarray:
    """b_e = 1.5 * ln(1/rank_e) with a seeded rank permutation of 1..n (fp32)."""
    rank = rank_permutation(seed, n)
    out = np.empty(n, dtype=np.float32)
    _get().synth_rank_bias(rank.ctypes.data, n, BIAS_SCALE, out.ctypes.data)
    return out


def route_logits(seed: int, T: int, N: int) -> np.ndarray:
    """Routing-only workload: fp32 logits = N(0,1) + b_e (one fp32 addition)."""
    noise = normal(seed, TID_LOGIT_NOISE, (T, N), 1.0, "f32")
    return (noise + router_bias(seed, N)[None, :]).astype(np.float32)


def layer_inputs(w: "Workload", seed: int = DEFAULT_SEED, with_experts: bool = True, n_shared: int = 0) -> dict:
    """All inputs of one MoGE layer workload as host arrays.

    Activations and weights are fp32 for an fp32 workload, else raw bf16 bits.
    The router bias is always fp32 (zero when the workload has no skew).  With
    n_shared > 0 the expert weights hold N + n_shared experts: the routed ones
    (the same values as without shared experts) followed by the shared ones.
    """
    dt = w.dtype
    T, d, N, I = w.T, w.d, w.N, w.I
    out = {
        "x": normal(seed, TID_X, (T, d), 1.0, dt),
        "w_router": normal(seed, TID_WR, (N, d), d ** -0.5, dt),
        "bias": router_bias(seed, N) if w.skew else np.zeros(N, dtype=np.float32),
    }
    if with_experts:
        E = N + n_shared
        out["w_gate"] = normal(seed, TID_WGATE, (E, I, d), d ** -0.5, dt)
        out["w_up"] = normal(seed, TID_WUP, (E, I, d), d ** -0.5, dt)
        out["w_down"] = normal(seed, TID_WDOWN, (E, d, I), I ** -0.5, dt)
    return out


def expert_weights(w: "Workload", e: int, seed: int = DEFAULT_SEED) -> tuple:
    """(W_gate[e], W_up[e], W_down[e]) alone, drawn from the same streams."""
    dt, d, I = w.dtype, w.d, w.I
    blk = I * d
    return (normal(seed, TID_WGATE, (I, d), d ** -0.5, dt, start=e * blk),
            normal(seed, TID_WUP, (I, d), d ** -0.5, dt, start=e * blk),
            normal(seed, TID_WDOWN, (d, I), I ** -0.5, dt, start=e * blk))


def study_scores(seed: int, b0: int, nb: int, T: int, N: int) -> np.ndarray:
    """Noise of batches [b0, b0+nb) of the imbalance Monte-Carlo study, [nb, T, N] fp32
    (Irwin-Hall sum of twelve 16-bit uniforms minus 6; exact, see synth.c).  The study's
    scores are this noise plus the router bias, one fp32 addition."""
    out = np.empty((nb, T, N), dtype=np.float32)
    _get().synth_study_scores(seed, TID_STUDY, b0, nb, T, N, out.ctypes.data)
    return out
