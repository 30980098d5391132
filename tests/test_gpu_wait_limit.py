"""A bounded wait that runs out on the GPU ends in a status code, not a hang.

Two grid barriers are made to run out: the fused small-problem kernels'
(between their phases) and the general path's dx'-product's (before it
reduces the partial sums). The fused small-problem kernels separate their
phases with grid barriers on a counter in the workspace. With BLR_FAULT=grid_barrier every barrier expects
one arrival more than the grid makes, so no barrier ever completes; with
BLR_WAIT_LIMIT_NS=1000000 each wait gives up after 1 ms. The kernels must then
record kStTimeoutGrid (0x40) in the workspace status word, leave their
remaining phases early (the abort flag ends the GEMM roles' waits), drain
what they issued, free their tensor memory and return: the calls complete,
the stream synchronises without a CUDA error, and the same process then runs
a normal forward+backward to parity. Nothing faults or traps.
"""
import numpy as np
import pytest
import torch

import oracle
from binary_rank_linear_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

K_ST_TIMEOUT_GRID = 0x40


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_grid_barrier_wait_runs_out_cleanly(monkeypatch):
    import binary_rank_linear_gb300 as blr
    from blr_gpu_run import run_layer
    t = wl.make_inputs(wl.WORKLOADS["tiny"])
    torch.cuda.synchronize()
    monkeypatch.setenv("BLR_SMALL_PATH", "fused")
    monkeypatch.setenv("BLR_FAULT", "grid_barrier")
    monkeypatch.setenv("BLR_WAIT_LIMIT_NS", "1000000")
    out = run_layer(t, gscale=0.0)  # forward and backward, both fused; check_status synchronises
    assert out["status"] & K_ST_TIMEOUT_GRID, f"status {out['status']:#x}"
    torch.cuda.synchronize()
    # the context is intact: the normal path runs to parity afterwards
    monkeypatch.delenv("BLR_FAULT")
    monkeypatch.delenv("BLR_WAIT_LIMIT_NS")
    monkeypatch.delenv("BLR_SMALL_PATH")
    good = run_layer(t, gscale=0.0)
    assert good["status"] == 0
    bu, bv = oracle.pack_signs(t["su"]), oracle.pack_signs(t["sv"])
    fw = oracle.forward(t["x"], bu, bv, t["g"], t["l"], t["h"])
    bw = oracle.backward(t["x"], t["dy"], bu, bv, t["g"], t["l"], t["h"])
    assert oracle.rel_err(good["y"], fw["y"]) <= 2e-3
    assert oracle.rel_err(good["dx"], bw["dx"]) <= 2e-3
    for k in ("dh", "dl", "dg"):
        assert oracle.rel_err(good[k], bw[k]) <= 5e-3
    assert np.isfinite(good["y"]).all()
    del blr


def test_folded_reduction_barrier_runs_out_cleanly(monkeypatch):
    """With BLR_REDUCE=fold the general path's dx'-product meets at a grid
    barrier before it reduces the partial sums of dh, dl and dg. With
    BLR_FAULT=grid_barrier
    that barrier expects one arrival more than the grid makes; under a 1 ms
    limit every CTA gives up, records kStTimeoutGrid and returns without
    reducing. The stream then synchronises cleanly and a normal pass runs to
    parity in the same process."""
    from blr_gpu_run import run_layer
    t = wl.make_inputs(wl.WORKLOADS["small"].with_shape(M=512))
    torch.cuda.synchronize()
    monkeypatch.setenv("BLR_REDUCE", "fold")
    monkeypatch.setenv("BLR_FAULT", "grid_barrier")
    monkeypatch.setenv("BLR_WAIT_LIMIT_NS", "1000000")
    out = run_layer(t, gscale=0.0)
    assert out["status"] & K_ST_TIMEOUT_GRID, f"status {out['status']:#x}"
    torch.cuda.synchronize()
    monkeypatch.delenv("BLR_FAULT")
    monkeypatch.delenv("BLR_WAIT_LIMIT_NS")
    good = run_layer(t, gscale=0.0)
    assert good["status"] == 0
    bu, bv = oracle.pack_signs(t["su"]), oracle.pack_signs(t["sv"])
    bw = oracle.backward(t["x"], t["dy"], bu, bv, t["g"], t["l"], t["h"])
    assert oracle.rel_err(good["dx"], bw["dx"]) <= 2e-3
    for k in ("dh", "dl", "dg"):
        assert oracle.rel_err(good[k], bw[k]) <= 5e-3
