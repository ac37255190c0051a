"""GPU parity of the layer with shared experts (moge_layer_forward_shared) against the oracle.

Every token visits every shared expert (weights at expert index N + s) and their SwiGLU outputs
are added with weight 1 to the gated routed combine.  Tolerances as for the layer:
max|y - ref| <= 2e-2 * max|ref| (bf16), 1e-5 (fp32); routing may differ only on near-ties.
"""
import numpy as np
import pytest
import torch

import oracle
import sparse_router_gemm_global_b300 as moge
import synth
from gpu_util import (DEV, config, expert_covering_tokens, host, max_rel_err, routing_mismatch_ok, torch_dtype,
                      upload_layer)
from synth import WORKLOADS

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-2, "f32": 1e-5}


def run_shared(w, d_inp, S):
    c = config(w)
    ws = moge.alloc_workspace(c, n_shared=S)
    out = {"y": torch.empty((w.T, w.d), dtype=torch_dtype(w), device=DEV),
           "topk_idx": torch.empty((w.T, w.K), dtype=torch.int32, device=DEV),
           "offsets": torch.empty(w.N + 1, dtype=torch.int32, device=DEV),
           "score": torch.empty(4, dtype=torch.float32, device=DEV)}
    aux = {k: v for k, v in out.items() if k != "y"}
    moge.moge_layer_forward_shared(c, S, d_inp["x"], d_inp["w_router"], d_inp["bias"], d_inp["w_gate"],
                                   d_inp["w_up"], d_inp["w_down"], out["y"], ws, aux=aux)
    torch.cuda.synchronize()
    assert moge.moge_query_device_status(ws) == 0
    return {k: host(v) for k, v in out.items()}


def check_shared(w, inp, got, S, tokens=None):
    ref = oracle.route(oracle.router_logits(inp["x"], inp["w_router"], inp["bias"]), w.M, w.kpg)
    near = routing_mismatch_ok(got["topk_idx"], ref["idx"], ref["p"], w.M, w.kpg)
    assert len(near) <= max(2, w.T // 1000)
    np.testing.assert_array_equal(got["offsets"], oracle.permute(got["topk_idx"], w.N)["offsets"])
    toks = np.arange(w.T) if tokens is None else np.asarray(tokens)
    toks = np.array([t for t in toks if t not in near], dtype=np.int32)
    y_ref = oracle.combine_tokens(toks, ref["idx"], ref["gate64"], inp["x"], inp["w_gate"], inp["w_up"],
                                  inp["w_down"])
    y_ref = y_ref + oracle.shared_experts_tokens(toks, w.N, S, inp["x"], inp["w_gate"], inp["w_up"], inp["w_down"])
    err = max_rel_err(got["y"][toks], y_ref)
    assert err <= TOL[w.dtype], f"{w.name} S={S}: max rel err {err:.3e}"
    return err


@pytest.mark.parametrize("T,d,N,M,kpg,I,S,dtype", [
    (64, 256, 16, 4, 1, 128, 2, "f32"),      # the tiny all-fp32 layer + 2 shared experts
    (1, 128, 16, 4, 2, 64, 4, "bf16"),       # one token
    (32, 4096, 64, 8, 2, 1408, 4, "bf16"),   # the decode layer + Pangu Pro's 4 shared experts
    (300, 256, 16, 4, 2, 192, 4, "bf16"),    # ragged rows, routed + shared segments
    (1100, 1024, 64, 8, 2, 256, 4, "bf16"),  # tokens-as-M tiles: each shared expert is one big segment
])
def test_shared_layer_matches_oracle(T, d, N, M, kpg, I, S, dtype):
    w = WORKLOADS["decode_t32"].with_(name=f"shared_{T}_{d}", T=T, d=d, N=N, M=M, kpg=kpg, I=I, dtype=dtype)
    inp = synth.layer_inputs(w, seed=T + d, n_shared=S)
    got = run_shared(w, upload_layer(inp), S)
    toks = None
    if T > 300:  # tokens reaching every tile of every routed expert and of every shared expert
        perm = oracle.permute(got["topk_idx"], w.N)
        toks, _ = expert_covering_tokens(perm["offsets"], perm["row_token"], w.T)
        toks = np.union1d(toks, np.arange(0, w.T, 128)).astype(np.int32)
    check_shared(w, inp, got, S, tokens=toks)


def test_zero_shared_experts_is_the_routed_layer_bit_for_bit():
    w = WORKLOADS["decode_t32"].with_(T=200, d=512, I=128)
    inp = synth.layer_inputs(w, seed=8)
    d_inp = upload_layer(inp)
    a = run_shared(w, d_inp, 0)
    c = config(w)
    ws = moge.alloc_workspace(c)
    y = torch.empty((w.T, w.d), dtype=torch.bfloat16, device=DEV)
    moge.moge_layer_forward(c, d_inp["x"], d_inp["w_router"], d_inp["bias"], d_inp["w_gate"], d_inp["w_up"],
                            d_inp["w_down"], y, ws)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(a["y"], host(y))
