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
