"""Failure detection of the bounded device waits, on the GPU, without any fault.

A small self-test kernel waits on mbarriers that nothing completes, through the same bounded
wait routine as the tensor-core kernels: one wait gives up after a short limit, raises the abort
flag and records MOGE_ERR_TIMEOUT in the workspace status word; the other leaves through the
abort flag.  The host reads the status, clears it, and the context keeps working.
"""
import time

import numpy as np
import pytest
import torch

import sparse_router_gemm_global_b300 as moge
import synth
from gpu_util import DEV, config, host, run_layer, upload_layer
from synth import WORKLOADS

pytestmark = pytest.mark.gpu

MOGE_ERR_TIMEOUT = 5


def test_bounded_wait_times_out_reports_and_recovers():
    w = WORKLOADS["decode_t32"].with_(T=40, d=256, I=128)
    c = config(w)
    ws = moge.alloc_workspace(c)
    res = torch.full((4,), 7, dtype=torch.int32, device=DEV)
    t0 = time.perf_counter()
    moge.moge_selftest_bounded_wait(ws, 20_000_000, res)   # 20 ms limit
    status = moge.moge_query_device_status(ws)             # synchronises the stream
    elapsed = time.perf_counter() - t0
    assert status == MOGE_ERR_TIMEOUT
    assert list(host(res)[:3]) == [0, 0, 1]                # both waits gave up; abort flag raised
    assert elapsed < 5.0                                   # bounded: nowhere near a hang
    moge.moge_reset_device_status(ws)
    assert moge.moge_query_device_status(ws) == 0
    # the context and the same workspace still run a layer correctly
    d_inp = upload_layer(synth.layer_inputs(w, seed=4))
    a = run_layer(w, d_inp, ws=ws)
    b = run_layer(w, d_inp)
    np.testing.assert_array_equal(a["y"], b["y"])


def test_selftest_rejects_bad_arguments():
    ws = torch.zeros(4096, dtype=torch.uint8, device=DEV)
    res = torch.zeros(4, dtype=torch.int32, device=DEV)
    with pytest.raises(moge.MoGEError):
        moge.moge_selftest_bounded_wait(ws, 0, res)
    with pytest.raises(moge.MoGEError):
        moge.moge_selftest_bounded_wait(ws, 2_000_000_000, res)
