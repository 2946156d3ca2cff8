"""Deferred status reporting: with gptq_set_status_mode(GPTQ_STATUS_DEFERRED) the calls
that otherwise synchronise to report device-side errors return once their work is
enqueued, and gptq_status_sync reports (and clears) the first such error."""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


def _npy(t):
    return t.detach().cpu().numpy()


def test_not_spd_is_reported_by_status_sync(lib):
    H = torch.tensor([[1.0, 2.0], [2.0, 1.0]], device="cuda")
    with lib.deferred_status():
        lib.status_sync()                      # nothing pending
        U, perm, dead = lib.gptq_prepare(H, None, 0.0)   # returns at once
        with pytest.raises(lib.GptqError) as e:
            lib.status_sync()
        assert e.value.status == 3
        lib.status_sync()                      # cleared
    # the synchronous default is back
    with pytest.raises(lib.GptqError):
        lib.gptq_prepare(H, None, 0.0)


def test_deferred_results_equal_synchronous(lib):
    d, rows = 384, 96
    spec = synth.XSpec(n=4 * d, d=d, kind="scaled", dtype="bf16", n_outliers=4, outlier_factor=20.0,
                       dead_frac=0.02, segment=1024)
    X = synth.make_x(spec, 11, device="cuda")
    W = synth.make_weight(rows, d, 0.02, 12, device="cuda")

    def layer():
        h = lib.Hessian(d)
        h.accumulate(X)
        H, diag, _ = h.finalize()
        U, perm, dead = lib.gptq_prepare(H, diag, 0.01, act_order=True)
        out = lib.gptq_quantize(W, U, perm, dead, 3, 128, False)
        torch.cuda.synchronize()
        return {k: _npy(v) for k, v in out.items()} | {"U": _npy(U)}

    ref = layer()
    with lib.deferred_status():
        got = layer()
        lib.status_sync()
    for k in ref:
        np.testing.assert_array_equal(got[k], ref[k], err_msg=k)


@pytest.mark.parametrize("d,rows,act", [(768, 200, False), (2176, 64, True)])
def test_cuda_graph_replay_equals_eager(lib, d, rows, act):
    """In deferred status mode the calls only enqueue work, so a whole prepare + quantize
    (two streams, programmatic dependent launches, events) can be captured into a CUDA
    graph; replays give the eager results bit for bit (d = 2176 also takes the
    super-panel schedule)."""
    spec = synth.XSpec(n=3 * d, d=d, kind="scaled", dtype="bf16", n_outliers=4, outlier_factor=20.0,
                       dead_frac=0.02, segment=1024)
    X = synth.make_x(spec, 21, device="cuda")
    W = synth.make_weight(rows, d, 0.02, 22, device="cuda")
    h = lib.Hessian(d)
    h.accumulate(X)
    H, diag, _ = h.finalize()
    prep_ws = torch.empty(lib.gptq_prepare_workspace_bytes(d, True), dtype=torch.uint8, device="cuda")

    def body():
        U, perm, dead = lib.gptq_prepare(H, diag, 0.01, act_order=act, ws=prep_ws)
        out = lib.gptq_quantize(W, U, perm, dead, 4, 128, True)
        out["U"] = U
        return out

    ref = body()
    torch.cuda.synchronize()
    ref = {k: _npy(v) for k, v in ref.items()}
    with lib.deferred_status():
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            body()
            lib.status_sync(s)
        torch.cuda.current_stream().wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            got = body()
        for _ in range(2):
            g.replay()
        lib.status_sync()
        torch.cuda.synchronize()
    for k in ref:
        np.testing.assert_array_equal(_npy(got[k]), ref[k], err_msg=k)
