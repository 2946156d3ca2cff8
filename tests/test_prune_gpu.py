"""GPU parity of pruning with GPTQ's update (GPTQ guide page, "Going further": SparseGPT reuses
the same update for pruning) against the oracle's `prune_layer`, given the oracle's U.

Protocol (the mask analogue of the code protocol):
  mask     the oracle runs teacher-forced: where the GPU's mask of a (row, block) differs
           from its own, the difference must be a near-tie of the saliency ranking (relative
           1e-4; fp32 saliencies of fp32 weights against fp64 ones), and the oracle then
           adopts the GPU's mask; at most 0.1% of (row, block) pairs may differ. Exactly
           round(sparsity * width) weights per row and block.
  Wp       pruned weights exactly 0; every weight within 1e-4 relative + 2e-5 max|W| absolute
           of the forced oracle's (fp32 accumulation of up to d compensation terms, 3xTF32
           trailing products at ~2^-20 relative each)
  row_loss sum err^2 within 1e-3 relative
  error    the relative output error tr(D S D^T) / tr(W S W^T) within 2% of a free-running
           oracle's
"""
import numpy as np
import pytest
import torch

import oracle as O
import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


def npy(t):
    return t.detach().cpu().numpy()


def _h_for(d, seed, n_mult=6):
    """H of correlated channels (X = Z A), every 37th channel exactly zero (dead)."""
    spec = synth.XSpec(n=n_mult * d, d=d, kind="correlated", dtype="bf16", segment=1024)
    X = synth.make_x(spec, seed, device=DEV)
    X[:, ::37] = 0
    Xh = synth.to_numpy_f64(X)
    S = O.xtx(Xh)
    return O.hessian_from_sum(S, Xh.shape[0]).astype(np.float32), np.diag(S).astype(np.float32), S


PCASES = [
    # rows, cols, sparsity, act_order
    (64, 256, 0.5, False),
    (96, 384, 0.25, True),
    (130, 640, 0.75, True),
    (33, 301, 0.5, False),     # cols % 4 != 0: the FFMA trailing update; ragged last block
    (200, 1100, 0.5, True),    # several super-blocks of the deferred trailing update
    (40, 256, 0.0, False),     # nothing pruned: W itself
    (40, 256, 1.0, False),     # everything pruned: zeros
]


@pytest.mark.parametrize("rows,cols,sparsity,act", PCASES)
def test_prune_given_oracle_u(lib, rows, cols, sparsity, act):
    H32, diag32, S = _h_for(cols, 700 + cols + rows)
    Uref, perm, dead = O.prepare(H32.astype(np.float64), 0.01, act, diag32.astype(np.float64))
    U32 = np.ascontiguousarray(Uref.astype(np.float32))
    W = synth.make_weight(rows, cols, 0.02, 800 + rows, device=DEV)
    Wh = synth.to_numpy_f64(W)
    out = lib.gptq_prune(W, torch.tensor(U32, device=DEV), torch.tensor(perm.astype(np.int32), device=DEV),
                         torch.tensor(dead.astype(np.uint8), device=DEV), sparsity)
    mask = npy(out["mask"]).astype(bool)
    Wp = npy(out["Wp"]).astype(np.float64)
    sp = float(np.float32(sparsity))
    ref = O.prune_layer(Wh, U32.astype(np.float64), perm, dead, sp, 128, forced_mask=mask)
    nblk = -(-cols // 128)
    assert len(ref["ties"]) <= 1e-3 * rows * nblk + 0.5, ref["ties"][:5]
    np.testing.assert_array_equal(mask, ref["mask"])
    # exactly round(sparsity * width) per row and block of loop positions
    for b0 in range(0, cols, 128):
        b1 = min(cols, b0 + 128)
        k = int(np.round(sp * (b1 - b0)))
        np.testing.assert_array_equal(mask[:, perm[b0:b1]].sum(axis=1), k)
    assert np.all(Wp[mask] == 0.0)
    np.testing.assert_allclose(Wp, ref["W"], rtol=1e-4, atol=2e-5 * np.abs(Wh).max())
    np.testing.assert_allclose(npy(out["row_loss"]), ref["err_sq"], rtol=1e-3, atol=1e-30)
    if 0.0 < sparsity < 1.0:
        free = O.prune_layer(Wh, U32.astype(np.float64), perm, dead, sp, 128)
        e_gpu = O.rel_output_error_from_xtx(S, Wh, Wp)
        e_ref = O.rel_output_error_from_xtx(S, Wh, free["W"])
        e_plain = O.rel_output_error_from_xtx(S, Wh, np.where(free["mask"], 0.0, np.where(dead, 0.0, Wh)))
        assert abs(e_gpu - e_ref) <= 0.02 * e_ref, (e_gpu, e_ref)
        assert e_gpu < e_plain   # the compensation helps on correlated inputs
    if sparsity == 0.0:
        np.testing.assert_array_equal(Wp, np.where(dead[None, :], 0.0, npy(W)))


def test_prune_rejects_bad_sparsity(lib):
    clib = lib.load()
    p = torch.zeros(16, device=DEV)
    ws = torch.empty(lib.gptq_prune_workspace_bytes(4, 4), dtype=torch.uint8, device=DEV)
    import ctypes
    for bad in (-0.1, 1.5, float("nan")):
        rc = clib.gptq_prune(ctypes.c_void_p(p.data_ptr()), 4, 4, ctypes.c_void_p(p.data_ptr()), None, None, bad,
                             ctypes.c_void_p(p.data_ptr()), None, None, ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                             None)
        assert rc == 1
