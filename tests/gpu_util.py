"""Helpers of the GPU parity tests: host arrays <-> device tensors, C-ABI calls.

Inputs always come from the ``synth`` generator; expected values always come
from ``oracle``.  Nothing here computes a layer result.
"""
from __future__ import annotations

import numpy as np
import torch

import sparse_router_gemm_global_b300 as moge

DEV = "cuda:0"


def dev(a: np.ndarray) -> torch.Tensor:
    """Host array -> device tensor (uint16 arrays are raw bf16 bits)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(DEV).view(torch.bfloat16)
    return torch.from_numpy(a).to(DEV)


def host(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def as_f64(a: np.ndarray) -> np.ndarray:
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def torch_dtype(w) -> torch.dtype:
    return torch.bfloat16 if w.dtype == "bf16" else torch.float32


def config(w, T=None):
    return moge.make_config(w.T if T is None else T, w.d, w.N, w.M, w.kpg, w.I, w.dtype)


def upload_layer(inp: dict) -> dict:
    return {k: dev(v) for k, v in inp.items()}


def run_layer(w, d_inp: dict, ws=None) -> dict:
    """moge_layer_forward with every aux output requested; returns host arrays."""
    c = config(w)
    ws = moge.alloc_workspace(c) if ws is None else ws
    T, N, K, M = w.T, w.N, w.K, w.M
    out = {
        "y": torch.empty((T, w.d), dtype=torch_dtype(w), device=DEV),
        "logits": torch.empty((T, N), dtype=torch.float32, device=DEV),
        "topk_idx": torch.empty((T, K), dtype=torch.int32, device=DEV),
        "topk_gate": torch.empty((T, K), dtype=torch.float32, device=DEV),
        "counts": torch.empty(N, dtype=torch.int32, device=DEV),
        "offsets": torch.empty(N + 1, dtype=torch.int32, device=DEV),
        "group_load": torch.empty(M, dtype=torch.int32, device=DEV),
        "score": torch.empty(4, dtype=torch.float32, device=DEV),
    }
    aux = {k: v for k, v in out.items() if k != "y"}
    moge.moge_layer_forward(c, d_inp["x"], d_inp["w_router"], d_inp["bias"], d_inp["w_gate"], d_inp["w_up"],
                            d_inp["w_down"], out["y"], ws, aux=aux)
    torch.cuda.synchronize()
    assert moge.moge_query_device_status(ws) == 0
    res = {k: host(v) for k, v in out.items()}
    res["score"] = res["score"][0]
    return res


def max_rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    """max |got - ref| / max |ref| (the layer's tolerance metric)."""
    g = as_f64(got) if got.dtype == np.uint16 else got.astype(np.float64)
    return float(np.max(np.abs(g - ref)) / max(np.max(np.abs(ref)), 1e-300))


def expert_covering_tokens(offsets, row_token, T, step=128):
    """Tokens whose rows reach every tile of every touched expert.

    For each expert e with rows [offsets[e], offsets[e+1]): its first row, its last row and the
    first row of every `step`-row block after the first (so both halves of every 256-row
    CTA-pair tile and every short last block are hit), mapped to tokens through row_token; plus
    tokens 0 and T-1.  Returns (sorted token array, number of touched experts)."""
    offsets = np.asarray(offsets, dtype=np.int64)
    rows = []
    touched = 0
    for e in range(len(offsets) - 1):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b <= a:
            continue
        touched += 1
        rows.extend(range(a, b, step))
        rows.append(b - 1)
    toks = set(int(row_token[r]) for r in rows)
    toks.update({0, T - 1})
    toks = np.array(sorted(toks), dtype=np.int32)
    return toks, touched


def routing_mismatch_ok(idx_gpu, idx_ref, p_ref, M, kpg, gap=1e-6):
    """Tokens whose routing differs from the oracle's.  Every differing slot must
    be a near-tie: the oracle's softmax probabilities of the two experts in that
    slot differ by less than `gap`.  Returns the set of such tokens."""
    bad = set()
    diff_t = np.nonzero(np.any(idx_gpu != idx_ref, axis=1))[0]
    for t in diff_t:
        for s_ in np.nonzero(idx_gpu[t] != idx_ref[t])[0]:
            a, b = int(idx_gpu[t, s_]), int(idx_ref[t, s_])
            assert abs(p_ref[t, a] - p_ref[t, b]) < gap, \
                f"token {t} slot {s_}: expert {a} vs {b}, probability gap {abs(p_ref[t, a] - p_ref[t, b]):.3g}"
        bad.add(int(t))
    return bad
