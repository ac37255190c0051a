"""The layer under CUDA graph capture.

One moge_layer_forward (or moge_layer_forward_shared) captured into a torch.cuda.CUDAGraph and
replayed gives the eager call's outputs bit for bit -- for the decode (weights-as-M, in-GEMM
gather), medium and tokens-as-M tile plans and the fp32 layer -- and again after new tokens are
copied into the captured input buffer.  The library makes no synchronising call and reads nothing
back to the host on the path, so a captured step replays without the host.
"""
import numpy as np
import pytest
import torch

import sparse_router_gemm_global_b300 as moge
import synth
from gpu_util import DEV, config, dev, host, torch_dtype, upload_layer
from synth import WORKLOADS

pytestmark = pytest.mark.gpu

CASES = {
    "decode": dict(),                                                      # T=32: swap32 + gather4
    "medium": dict(T=300, d=512, I=256),                                   # 64-token weights-as-M tiles
    "pairs": dict(T=2048, d=1024, I=512),                                  # CTA-pair tokens-as-M tiles
    "fp32": dict(T=64, d=256, N=16, M=4, kpg=1, I=128, dtype="f32"),       # CUDA-core path
}


def outputs(w):
    T, N, K, M = w.T, w.N, w.K, w.M
    return {
        "y": torch.empty((T, w.d), dtype=torch_dtype(w), device=DEV),
        "topk_idx": torch.empty((T, K), dtype=torch.int32, device=DEV),
        "topk_gate": torch.empty((T, K), dtype=torch.float32, device=DEV),
        "counts": torch.empty(N, dtype=torch.int32, device=DEV),
        "group_load": torch.empty(M, dtype=torch.int32, device=DEV),
        "score": torch.empty(4, dtype=torch.float32, device=DEV),
    }


def poison(out):
    for v in out.values():
        v.fill_(-3 if v.dtype == torch.int32 else float("nan"))


def call(c, S, d, out, ws):
    aux = {k: v for k, v in out.items() if k != "y"}
    if S:
        moge.moge_layer_forward_shared(c, S, d["x"], d["w_router"], d["bias"], d["w_gate"], d["w_up"],
                                       d["w_down"], out["y"], ws, aux=aux)
    else:
        moge.moge_layer_forward(c, d["x"], d["w_router"], d["bias"], d["w_gate"], d["w_up"], d["w_down"],
                                out["y"], ws, aux=aux)


def snapshot(out):
    res = {k: host(v) for k, v in out.items()}
    res["score"] = res["score"][:1]  # one float; the buffer is padded to 16 bytes
    return res


@pytest.mark.parametrize("case", list(CASES))
@pytest.mark.parametrize("S", [0, 4])
@pytest.mark.parametrize("mode", ["global", "thread_local"])
def test_graph_replay_matches_eager(case, S, mode):
    w = WORKLOADS["decode_t32"].with_(**CASES[case])
    d = upload_layer(synth.layer_inputs(w, seed=70, n_shared=S))
    c = config(w)
    ws = moge.alloc_workspace(c, n_shared=S)
    eager = outputs(w)
    call(c, S, d, eager, ws)
    torch.cuda.synchronize()
    ref = snapshot(eager)

    out = outputs(w)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode=mode):
        call(c, S, d, out, ws)
    for _ in range(3):
        poison(out)
        g.replay()
    torch.cuda.synchronize()
    got = snapshot(out)
    for k in ref:
        np.testing.assert_array_equal(got[k], ref[k], err_msg=k)

    # new tokens in the captured input buffer: the replay follows them
    x2 = synth.layer_inputs(w.with_(name=w.name + "_x2"), seed=71, with_experts=False)["x"]
    d["x"].copy_(dev(x2))
    call(c, S, d, eager, ws)
    torch.cuda.synchronize()
    ref2 = snapshot(eager)
    poison(out)
    g.replay()
    torch.cuda.synchronize()
    got2 = snapshot(out)
    for k in ref2:
        np.testing.assert_array_equal(got2[k], ref2[k], err_msg=k)
    assert not np.array_equal(ref2["y"], ref["y"])
    assert moge.moge_query_device_status(ws) == 0
