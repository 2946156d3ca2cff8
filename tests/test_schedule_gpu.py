"""The benchmark's concurrent schedules (the groups' gptq_prepare calls, or their prepare and
quantize calls, side by side on their own streams) give the serial schedule's outputs bit for
bit. With 2048 tokens per input every Hessian tile takes exactly one accumulation into a
zeroed S, so H itself is bit-reproducible and the comparison can be exact."""
import numpy as np
import pytest
import torch

import bench

pytestmark = pytest.mark.gpu


def _snap(outs):
    torch.cuda.synchronize()
    return [{k: v.detach().cpu().numpy().copy() for k, v in o.items()} for o in outs]


def test_concurrent_schedules_equal_serial(lib):
    args = bench.parse(["--config", "4", "--x-tokens", "2048", "--bits", "4"])
    wl, layers = bench.build_layers(4, "cuda", wl=bench.workload_for(args))
    runner = bench.Runner(lib, layers, torch.device("cuda"))
    ref = _snap(runner.step())
    for in_group, fork in ((False, False), (True, False), (True, True)):
        with lib.deferred_status():
            got = _snap(runner.step_concurrent(quantize_in_group=in_group, fork_layers=fork))
            lib.status_sync()
        for li, (a, b) in enumerate(zip(got, ref)):
            for k in b:
                np.testing.assert_array_equal(a[k], b[k], err_msg=f"layer {li} {k} (in_group={in_group}, fork={fork})")


def test_layer_fork_with_shared_input_equals_serial(lib):
    """Two bit widths on each input: the layers of a group quantise on their own streams and
    workspaces at the same time, against the same U; each gives its serial result."""
    args = bench.parse(["--config", "4", "--x-tokens", "2048"])
    wl, layers = bench.build_layers(4, "cuda", wl=bench.workload_for(args))
    layers = [L for L in layers if L.spec.q.bits in (2, 4) and L.X.shape[1] == 4096]
    runner = bench.Runner(lib, layers, torch.device("cuda"))
    assert max(len(g) for g in runner.groups) == 2
    ref = _snap(runner.step())
    with lib.deferred_status():
        got = _snap(runner.step_concurrent(quantize_in_group=True, fork_layers=True))
        lib.status_sync()
    for li, (a, b) in enumerate(zip(got, ref)):
        for k in b:
            np.testing.assert_array_equal(a[k], b[k], err_msg=f"layer {li} {k}")


def test_schedules_with_copy_events_equal_serial(lib):
    """The e2e form of the step: inputs and weights copied on a side stream, each input one
    chunk whose event its Hessian waits on, weights behind events, a done event per layer,
    the groups in a different order. Every schedule gives the plain serial outputs."""
    args = bench.parse(["--config", "4", "--x-tokens", "2048", "--bits", "3"])
    wl, layers = bench.build_layers(4, "cuda", wl=bench.workload_for(args))
    runner = bench.Runner(lib, layers, torch.device("cuda"))
    ref = _snap(runner.step())
    side = torch.cuda.Stream()
    Xs = {id(L.X): torch.empty_like(L.X) for L in layers}
    dX = [Xs[id(L.X)] for L in layers]
    dW = [torch.empty_like(L.Wcat) for L in layers]
    x_chunks = {gi: [(dX[g[0]], torch.cuda.Event(), 0)] for gi, g in enumerate(runner.groups)}
    w_ready = [torch.cuda.Event() for _ in layers]
    layer_done = [torch.cuda.Event() for _ in layers]
    order = list(reversed(range(len(runner.groups))))
    for sched in ("serial", "prepare", "groups", "layers"):
        for x in dX:
            x.zero_()
        torch.cuda.synchronize()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for gi in order:
                g = runner.groups[gi]
                dX[g[0]].copy_(layers[g[0]].X)
                x_chunks[gi][0][1].record()
                for li in g:
                    dW[li].copy_(layers[li].Wcat)
                    w_ready[li].record()
        kw = dict(Xs=dX, Wcats=dW, x_chunks=x_chunks, w_ready=w_ready, layer_done=layer_done, order=order)
        with lib.deferred_status():
            outs = (runner.step(**kw) if sched == "serial"
                    else runner.step_concurrent(quantize_in_group=(sched != "prepare"),
                                                fork_layers=(sched == "layers"), **kw))
            for ev in layer_done:
                ev.synchronize()
            got = _snap(outs)
            lib.status_sync()
        for li, (a, b) in enumerate(zip(got, ref)):
            for k in b:
                np.testing.assert_array_equal(a[k], b[k], err_msg=f"layer {li} {k} ({sched})")
