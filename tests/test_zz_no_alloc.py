"""gptq_prepare_noalloc, the allocation-free variant of gptq_prepare.

It serves callers that cannot allocate device memory themselves (a host framework that
owns all device memory, or a path that cannot take cudaMalloc's implicit
synchronisation): its scratch is a fixed array inside the library. This file is named
so that pytest collects it last; it must pass alone in a fresh process and after the
other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


def _inputs(lib, d, seed):
    spec = synth.XSpec(n=3 * d, d=d, kind="scaled", dtype="bf16", n_outliers=4, outlier_factor=20.0,
                       dead_frac=0.02, segment=1024)
    X = synth.make_x(spec, seed, device="cuda")
    h = lib.Hessian(d)
    h.accumulate(X)
    H, diag, _ = h.finalize()
    return H, diag


def _noalloc(clib, H, diag, d, damp, act_order):
    U = torch.empty(d, d, dtype=torch.float32, device="cuda")
    perm = torch.empty(d, dtype=torch.int32, device="cuda")
    dead = torch.empty(d, dtype=torch.uint8, device="cuda")
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = clib.gptq_prepare_noalloc(ctypes.c_void_p(H.data_ptr()), ctypes.c_void_p(diag.data_ptr()), d,
                                   ctypes.c_float(damp), 1 if act_order else 0, ctypes.c_void_p(U.data_ptr()),
                                   ctypes.c_void_p(perm.data_ptr()), ctypes.c_void_p(dead.data_ptr()), s)
    return rc, U, perm, dead


def test_prepare_noalloc_matches_prepare_on_two_calls(lib):
    clib = lib.load()
    # two calls in a row, different sizes and options: the shared scratch keeps the first
    # call's contents, which must not leak into the second
    for d, act_order, seed in ((1000, True, 5), (768, False, 6)):
        H, diag = _inputs(lib, d, seed)
        rc, U, perm, dead = _noalloc(clib, H, diag, d, 0.01, act_order)
        assert rc == 0, lib.gptq_status_string(rc)
        Ur, pr, dr = lib.gptq_prepare(H, diag, 0.01, act_order=act_order)
        torch.cuda.synchronize()
        a, b = U.double().cpu().numpy(), Ur.double().cpu().numpy()
        assert np.linalg.norm(a - b) / np.linalg.norm(b) <= 1e-4
        assert torch.equal(perm, pr)
        assert torch.equal(dead, dr)


def test_prepare_noalloc_rejects_sizes_beyond_its_scratch(lib):
    clib = lib.load()
    d = 1025
    H = torch.eye(d, device="cuda")
    rc, _, _, _ = _noalloc(clib, H, torch.ones(d, device="cuda"), d, 0.01, False)
    assert rc == 2   # GPTQ_ERR_UNSUPPORTED
