"""GPU parity of the layer added to a residual stream (moge_layer_forward_residual) against the
oracle: y = r + sum_k gate_k FFN_k(x) + sum_s FFN_s(x), the residual row added once, unweighted.

The residual is drawn with the magnitude of the layer's own output, so that its error budget and
the FFN's are of one size; tolerance as for the layer, max|y - ref| <= 2e-2 * max|ref| (bf16),
1e-5 (fp32), on tokens whose routing is not a near-tie.  The in-place form (y is the residual
buffer) must equal the out-of-place one bit for bit, and a zero residual the plain layer.
"""
import numpy as np
import pytest
import torch

import oracle
import sparse_router_gemm_global_b300 as moge
import synth
from gpu_util import DEV, as_f64, config, dev, host, max_rel_err, routing_mismatch_ok, torch_dtype, upload_layer
from synth import WORKLOADS

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-2, "f32": 1e-5}


def forward(w, d, S, residual, y):
    c = config(w)
    ws = moge.alloc_workspace(c, n_shared=S)
    idx = torch.empty((w.T, w.K), dtype=torch.int32, device=DEV)
    moge.moge_layer_forward_residual(c, S, d["x"], residual, d["w_router"], d["bias"], d["w_gate"], d["w_up"],
                                     d["w_down"], y, ws, aux={"topk_idx": idx})
    torch.cuda.synchronize()
    assert moge.moge_query_device_status(ws) == 0
    return host(y), host(idx)


@pytest.mark.parametrize("T,d,N,M,kpg,I,S,dtype", [
    (32, 4096, 64, 8, 2, 1408, 4, "bf16"),   # the decode layer + 4 shared experts
    (300, 256, 16, 4, 2, 192, 4, "bf16"),    # weights-as-M tiles
    (1100, 1024, 64, 8, 2, 256, 0, "bf16"),  # CTA-pair tiles, no shared expert
    (64, 256, 16, 4, 1, 128, 2, "f32"),      # the all-fp32 layer
])
def test_residual_layer_matches_oracle(T, d, N, M, kpg, I, S, dtype):
    w = WORKLOADS["decode_t32"].with_(name=f"res_{T}", T=T, d=d, N=N, M=M, kpg=kpg, I=I, dtype=dtype)
    inp = synth.layer_inputs(w, seed=90 + T, n_shared=S)
    d_inp = upload_layer(inp)
    # a residual of the layer output's own scale
    scale = float(np.max(np.abs(oracle.layer_forward(inp["x"], inp["w_router"], inp["bias"], inp["w_gate"],
                                                     inp["w_up"], inp["w_down"], M, kpg, tokens=[0, 1],
                                                     n_shared=S)["y"])))
    r = synth.normal(91 + T, synth.TID_X, (T, d), scale, dtype)
    y, idx = forward(w, d_inp, S, dev(r), torch.empty((T, d), dtype=torch_dtype(w), device=DEV))

    ref = oracle.route(oracle.router_logits(inp["x"], inp["w_router"], inp["bias"]), M, kpg)
    near = routing_mismatch_ok(idx, ref["idx"], ref["p"], M, kpg)
    assert len(near) <= max(2, T // 1000)
    toks = np.array([t for t in range(T) if t not in near], dtype=np.int32)
    y_ref = oracle.layer_forward(inp["x"], inp["w_router"], inp["bias"], inp["w_gate"], inp["w_up"],
                                 inp["w_down"], M, kpg, tokens=toks, n_shared=S, residual=r)["y"]
    err = max_rel_err(y[toks], y_ref)
    assert err <= TOL[dtype], f"max rel err {err:.3e}"

    # in place: y is the residual buffer
    buf = dev(r)
    y2, _ = forward(w, d_inp, S, buf, buf)
    np.testing.assert_array_equal(y2, y)

    # a zero residual gives the plain layer's values
    zeros = torch.zeros((T, d), dtype=torch_dtype(w), device=DEV)
    y0, _ = forward(w, d_inp, S, zeros, torch.empty_like(zeros))
    c = config(w)
    ws = moge.alloc_workspace(c, n_shared=S)
    plain = torch.empty_like(zeros)
    moge.moge_layer_forward_shared(c, S, d_inp["x"], d_inp["w_router"], d_inp["bias"], d_inp["w_gate"],
                                   d_inp["w_up"], d_inp["w_down"], plain, ws)
    torch.cuda.synchronize()
    yp = host(plain)
    np.testing.assert_array_equal(as_f64(y0) if y0.dtype == np.uint16 else y0,
                                  as_f64(yp) if yp.dtype == np.uint16 else yp)
