"""Concurrent layer calls on separate streams.

The library keeps no per-call state outside the caller's workspace (routing tickets, status word,
permutation scratch all live there), so two moge_layer_forward calls running at the same time on
two streams with two workspaces give exactly the outputs each gives alone.
"""
import numpy as np
import pytest
import torch

import sparse_router_gemm_global_b300 as moge
import synth
from gpu_util import DEV, config, host, torch_dtype, upload_layer
from synth import WORKLOADS

pytestmark = pytest.mark.gpu

SHAPES = {
    "decode": dict(T=32),                     # small router + gather4 GEMM
    "medium": dict(T=300, d=512, I=256),      # tensor-core router, 128-token tiles
    "pairs": dict(T=2048, d=1024, I=512),     # CTA-pair tiles
}


def outputs(w):
    return {"y": torch.empty((w.T, w.d), dtype=torch_dtype(w), device=DEV),
            "topk_idx": torch.empty((w.T, w.K), dtype=torch.int32, device=DEV),
            "counts": torch.empty(w.N, dtype=torch.int32, device=DEV)}


def call(c, d, out, ws, stream=None):
    moge.moge_layer_forward(c, d["x"], d["w_router"], d["bias"], d["w_gate"], d["w_up"], d["w_down"], out["y"],
                            ws, aux={k: v for k, v in out.items() if k != "y"}, stream=stream)


@pytest.mark.parametrize("a,b", [("decode", "pairs"), ("medium", "medium"), ("pairs", "pairs")])
def test_two_streams_match_sequential_calls(a, b):
    wa = WORKLOADS["decode_t32"].with_(name="sa", **SHAPES[a])
    wb = WORKLOADS["decode_t32"].with_(name="sb", **SHAPES[b])
    da = upload_layer(synth.layer_inputs(wa, seed=80))
    db = upload_layer(synth.layer_inputs(wb, seed=81))
    ca, cb = config(wa), config(wb)
    wsa, wsb = moge.alloc_workspace(ca), moge.alloc_workspace(cb)
    ref_a, ref_b = outputs(wa), outputs(wb)
    call(ca, da, ref_a, wsa)
    call(cb, db, ref_b, wsb)
    torch.cuda.synchronize()
    ref_a = {k: host(v) for k, v in ref_a.items()}
    ref_b = {k: host(v) for k, v in ref_b.items()}

    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    out_a, out_b = outputs(wa), outputs(wb)
    torch.cuda.synchronize()
    for _ in range(5):  # interleave launches of the two streams
        call(ca, da, out_a, wsa, stream=sa)
        call(cb, db, out_b, wsb, stream=sb)
    torch.cuda.synchronize()
    for k in ref_a:
        np.testing.assert_array_equal(host(out_a[k]), ref_a[k], err_msg=f"a:{k}")
        np.testing.assert_array_equal(host(out_b[k]), ref_b[k], err_msg=f"b:{k}")
    assert moge.moge_query_device_status(wsa) == 0 and moge.moge_query_device_status(wsb) == 0
