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


def test_nonfinite_inputs_are_reported(lib):
    """A NaN or an infinity written into host-side inputs is reported as GPTQ_ERR_NONFINITE
    (7): in X by gptq_hessian_finalize (through diag(S)), in H by gptq_prepare, in W by
    gptq_quantize and rtn_quantize; a NaN in a dead column is never read. Clean calls on the
    same objects then succeed."""
    d, rows, n = 256, 48, 1024
    spec = synth.XSpec(n=n, d=d, kind="scaled", dtype="bf16", n_outliers=2, outlier_factor=20.0,
                       dead_frac=0.05, segment=1024)
    Xh = synth.make_x(spec, 51, device="cpu")
    Wh = synth.make_weight(rows, d, 0.02, 52, device="cpu")
    X = Xh.cuda()
    W = Wh.cuda()

    # X: a NaN in one token, an infinity in another
    for bad in (float("nan"), float("inf")):
        Xb = Xh.clone()
        Xb[17, 33] = bad
        h = lib.Hessian(d)
        h.accumulate(Xb.cuda())
        with pytest.raises(lib.GptqError) as e:
            h.finalize()
        assert e.value.status == 7
        h.reset()                      # the accumulator is usable again after a reset
        h.accumulate(X)
        h.finalize()

    h = lib.Hessian(d)
    h.accumulate(X)
    H, diag, _ = h.finalize()
    # H: one entry of the upper triangle, then one on the diagonal
    for (i, j) in ((3, 100), (5, 5)):
        Hb = H.clone()
        Hb[i, j] = float("nan")
        with pytest.raises(lib.GptqError) as e:
            lib.gptq_prepare(Hb, diag, 0.01)
        assert e.value.status == 7
    U, perm, dead = lib.gptq_prepare(H, diag, 0.01)
    dead_cols = np.nonzero(_npy(dead))[0]
    assert len(dead_cols) > 0

    # W: a live entry (NaN, then -inf) fails both quantizers
    for bad in (float("nan"), float("-inf")):
        Wb = Wh.clone()
        live = int(np.setdiff1d(np.arange(d), dead_cols)[7])
        Wb[4, live] = bad
        Wb = Wb.cuda()
        with pytest.raises(lib.GptqError) as e:
            lib.gptq_quantize(Wb, U, perm, dead, 4, 128, True)
        assert e.value.status == 7
        with pytest.raises(lib.GptqError) as e:
            lib.rtn_quantize(Wb, 4, 128, True, dead=dead)
        assert e.value.status == 7
    # a NaN in a dead column is zeroed, never read
    Wd = Wh.clone()
    Wd[:, int(dead_cols[0])] = float("nan")
    ref = lib.gptq_quantize(W, U, perm, dead, 4, 128, True)
    got = lib.gptq_quantize(Wd.cuda(), U, perm, dead, 4, 128, True)
    np.testing.assert_array_equal(_npy(got["codes"]), _npy(ref["codes"]))
    lib.rtn_quantize(Wd.cuda(), 4, 128, True, dead=dead)
    # U not finite on its diagonal
    Ub = U.clone()
    Ub[9, 9] = float("inf")
    with pytest.raises(lib.GptqError) as e:
        lib.gptq_quantize(W, Ub, perm, dead, 4, 128, True)
    assert e.value.status == 7


def test_bounded_waits_time_out_and_unwind(lib):
    """With the library's test hook the pipeline waits of every tensor-core kernel get a
    limit of 0 (give up at the first wait that is not already complete): the Hessian, the
    trailing-update GEMM inside gptq_quantize and the stored-form consumer then report
    GPTQ_ERR_TIMEOUT (5) after unwinding (in-flight copies and MMAs drained with the full
    limit, TMEM freed). With the limit restored, the same calls give the results they gave
    before."""
    clib = lib.load()
    d, rows, n = 512, 256, 8192
    spec = synth.XSpec(n=n, d=d, kind="scaled", dtype="bf16", n_outliers=4, outlier_factor=20.0, segment=2048)
    X = synth.make_x(spec, 61, device="cuda")
    W = synth.make_weight(rows, d, 0.02, 62, device="cuda")

    def hessian():
        h = lib.Hessian(d)
        h.accumulate(X)
        return h.finalize()[:2]

    def downstream(H, diag):
        U, perm, dead = lib.gptq_prepare(H, diag, 0.01)
        out = lib.gptq_quantize(W, U, perm, dead, 4, 128, True)
        Y = lib.gptq_dequant_matmul(X[:1024].contiguous(), out["packed"], out["scales"], out["zeros"], out["g_idx"], 4)
        torch.cuda.synchronize()
        return {"U": _npy(U), "codes": _npy(out["codes"]), "Y": _npy(Y)}, (U, perm, dead, out)

    H, diag = hessian()
    H_ref = _npy(H)
    ref, (U, perm, dead, out) = downstream(H, diag)
    try:
        assert clib.gptq_test_set_wait_limit_ns(0) == 0
        h = lib.Hessian(d)
        h.accumulate(X)
        with pytest.raises(lib.GptqError) as e:
            h.finalize()
        assert e.value.status == 5
        with pytest.raises(lib.GptqError) as e:
            lib.gptq_quantize(W, U, perm, dead, 4, 128, True)
        assert e.value.status == 5
        with pytest.raises(lib.GptqError) as e:
            lib.gptq_dequant_matmul(X[:1024].contiguous(), out["packed"], out["scales"], out["zeros"], out["g_idx"], 4)
        assert e.value.status == 5
    finally:
        assert clib.gptq_test_set_wait_limit_ns(2_000_000_000) == 0
    # the Hessian's fp32 atomics add the CTAs' partial sums in a run-dependent order: the
    # same H to rounding; given the same H, the rest is deterministic and bit-identical
    H2, _ = hessian()
    assert np.linalg.norm(_npy(H2) - H_ref) <= 1e-6 * np.linalg.norm(H_ref)
    got, _ = downstream(H, diag)
    for k in ref:
        np.testing.assert_array_equal(got[k], ref[k], err_msg=k)


def test_dequant_matmul_in_cuda_graph(lib):
    """The stored-form consumer allocates nothing and copies nothing from the host, so in
    deferred status mode it can be captured into a CUDA graph; replays (both the grouped
    and the scattered-group kernel) give the eager results bit for bit."""
    d, rows, n = 384, 256, 2048
    spec = synth.XSpec(n=n, d=d, kind="scaled", dtype="bf16", n_outliers=4, outlier_factor=20.0, segment=2048)
    X = synth.make_x(spec, 71, device="cuda")
    W = synth.make_weight(rows, d, 0.02, 72, device="cuda")
    h = lib.Hessian(d)
    h.accumulate(X)
    H, diag, _ = h.finalize()
    for act in (False, True):
        U, perm, dead = lib.gptq_prepare(H, diag, 0.01, act_order=act)
        st = lib.gptq_quantize(W, U, perm, dead, 3, 128, True)
        Xs = X[:512].contiguous()
        Y = torch.empty(512, rows, dtype=torch.float32, device="cuda")

        def body():
            lib.gptq_dequant_matmul(Xs, st["packed"], st["scales"], st["zeros"], st["g_idx"], 3, out=Y)

        body()
        torch.cuda.synchronize()
        ref = _npy(Y)
        with lib.deferred_status():
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                body()
                lib.status_sync(s)
            torch.cuda.current_stream().wait_stream(s)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                body()
            Y.zero_()
            for _ in range(2):
                g.replay()
            lib.status_sync()
            torch.cuda.synchronize()
        np.testing.assert_array_equal(_npy(Y), ref)
