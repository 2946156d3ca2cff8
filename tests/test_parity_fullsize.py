"""Full-size parity for the large workloads, on the inputs and call sequence bench.py times.

At these sizes the oracle checks samples it can compute one by one:
  H      sampled entries 2/n sum_t X[t,i] X[t,j] in fp64 from the same bf16 bits,
         |dH_ij| <= 1e-5 * sqrt(H_ii H_jj)
  U      the oracle's inv + Cholesky (fp64) of the GPU's H: relative Frobenius <= 1e-4
  codes  a sample of rows (rows are independent given U) through the teacher-forced
         oracle loop given the GPU's U: >= 99.99% identical, mismatches only at half-points
  error  the sampled rows' relative output error tr(D S D^T) / tr(W S W^T) within 2% of a
         free-running oracle's on the same rows
(GPTQ below RTN is not asserted here: with independent channels and n/d = 64 the Hessian
is close to diagonal, and the oracle itself lands at or slightly above RTN on these rows;
the claim is checked where it holds, in test_parity_gpu.)
  packed codes and g_idx bit-exact given the codes
"""
import numpy as np
import pytest
import torch

import bench
import oracle as O
import synth

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def npy(t):
    return t.detach().cpu().numpy()


def _check_hessian(X, H, diag, n, rng, npairs=48):
    d = X.shape[1]
    Hd = npy(torch.diagonal(H)).astype(np.float64)
    cols = np.unique(np.concatenate([rng.choice(d, npairs, replace=False), np.argsort(-Hd)[:4]]))
    Xs = synth.to_numpy_f64(X[:, torch.as_tensor(cols, device=X.device)])
    S = Xs.T @ Xs
    Href = 2.0 * S / n
    Hg = npy(H[torch.as_tensor(cols, device=H.device)][:, torch.as_tensor(cols, device=H.device)]).astype(np.float64)
    scale = np.sqrt(np.outer(np.diag(Href), np.diag(Href)))
    ok = scale > 0
    assert np.all(np.abs(Hg - Href)[ok] <= 1e-5 * scale[ok])
    assert np.all(Hg[~ok] == 0)
    np.testing.assert_allclose(npy(diag)[cols], np.diag(S), rtol=2e-5)


def _layer(lib, L, rng, row_sample, check_u=True):
    q = L.spec.q
    X = L.X
    n, d = X.shape
    h = lib.Hessian(d)
    h.accumulate(X)
    H, diag, nn = h.finalize()
    assert nn == n
    _check_hessian(X, H, diag, n, rng)
    U, perm, dead = lib.gptq_prepare(H, diag, q.damp, act_order=q.act_order)
    H64 = npy(H).astype(np.float64)
    diag64 = npy(diag).astype(np.float64)
    Ug = npy(U).astype(np.float64)
    if check_u:
        Uref, pref, dref = O.prepare(H64, q.damp, q.act_order, diag64)
        assert np.linalg.norm(Ug - Uref) / np.linalg.norm(Uref) <= 1e-4
        del Uref
    else:
        dref = O.dead_mask(H64)
        pref = O.act_order_perm(diag64) if q.act_order else np.arange(d)
    np.testing.assert_array_equal(npy(perm), pref)
    np.testing.assert_array_equal(npy(dead).astype(bool), dref)
    S = H64 * (n / 2.0)
    outs = []
    for W in L.Ws:
        out = lib.gptq_quantize(W, U, perm, dead, q.bits, q.group, q.sym)
        rtn = lib.rtn_quantize(W, q.bits, q.group, q.sym, dead=dead)
        rows = np.sort(rng.choice(W.shape[0], min(row_sample, W.shape[0]), replace=False))
        ri = torch.as_tensor(rows, device=W.device)
        Wr = synth.to_numpy_f64(W[ri])
        codes = npy(out["codes"][ri]).astype(np.int64)
        zeros = npy(out["zeros"][ri]).astype(np.int64)
        forced = O.gptq_quantize(Wr, Ug, pref, dref, q.bits, q.group, q.sym, forced_codes=codes,
                                 forced_zeros=None if q.sym else zeros)
        nmis = len([t for t in forced["ties"] if t[2] == "code"])
        assert nmis <= 1e-4 * codes.size + 0.5, forced["ties"][:5]
        np.testing.assert_allclose(npy(out["scales"][ri]), forced["scales"], rtol=2e-5)
        np.testing.assert_array_equal(npy(out["packed"][ri]).view(np.uint32), forced["packed"])
        np.testing.assert_array_equal(npy(out["g_idx"]), forced["g_idx"])
        free = O.gptq_quantize(Wr, Ug, pref, dref, q.bits, q.group, q.sym)
        e_gpu = O.rel_output_error_from_xtx(S, Wr, npy(out["Wq"][ri]))
        e_ref = O.rel_output_error_from_xtx(S, Wr, free["Wq"])
        e_rtn = O.rel_output_error_from_xtx(S, Wr, npy(rtn["Wq"][ri]))
        assert abs(e_gpu - e_ref) <= 0.02 * e_ref, (e_gpu, e_ref)
        print(f"rows={len(rows)} bits={q.bits} rel output error: gpu {e_gpu:.6f} oracle {e_ref:.6f} rtn {e_rtn:.6f}")
        outs.append((e_gpu, e_ref, e_rtn))
    return outs


def test_llama7b_attention_projection(lib):
    wl, layers = bench.build_layers(2, "cuda")
    rng = np.random.default_rng(2)
    _layer(lib, layers[0], rng, row_sample=256)


def test_llama7b_attention_end_to_end_from_oracle_chain(lib):
    """One comparison over the whole chain at full size: the oracle's own fp64 H (streamed
    over all 262144 tokens from the same bf16 bits), its own inv + Cholesky U, and its
    free-running loop on a sample of rows, against the GPU's Hessian -> prepare -> quantize
    of the same layer; the sampled rows' relative output error (through the oracle's S)
    within 2%."""
    wl, layers = bench.build_layers(2, "cuda")
    L = layers[0]
    q = L.spec.q
    X, W = L.X, L.Ws[0]
    n, d = X.shape
    S = None
    for r in range(0, n, 8192):
        Xb = synth.to_numpy_f64(X[r:r + 8192])
        S = O.xtx(Xb) if S is None else S + O.xtx(Xb)
    Href = O.hessian_from_sum(S, n)
    Uref, pref, dref = O.prepare(Href, q.damp, q.act_order, np.diag(S))
    h = lib.Hessian(d)
    h.accumulate(X)
    H, diag, _ = h.finalize()
    U, perm, dead = lib.gptq_prepare(H, diag, q.damp, act_order=q.act_order)
    out = lib.gptq_quantize(W, U, perm, dead, q.bits, q.group, q.sym)
    rng = np.random.default_rng(22)
    rows = np.sort(rng.choice(W.shape[0], 128, replace=False))
    ri = torch.as_tensor(rows, device=W.device)
    Wr = synth.to_numpy_f64(W[ri])
    ref = O.gptq_quantize(Wr, Uref, pref, dref, q.bits, q.group, q.sym)
    e_gpu = O.rel_output_error_from_xtx(S, Wr, npy(out["Wq"][ri]))
    e_ref = O.rel_output_error_from_xtx(S, Wr, ref["Wq"])
    print(f"end to end from the oracle's H and U: gpu {e_gpu:.6f} oracle {e_ref:.6f}")
    assert abs(e_gpu - e_ref) <= 0.02 * e_ref, (e_gpu, e_ref)
    np.testing.assert_array_equal(npy(perm), pref)
    np.testing.assert_array_equal(npy(dead).astype(bool), dref)


def test_mlp_down_projection_act_order(lib):
    wl, layers = bench.build_layers(3, "cuda")
    rng = np.random.default_rng(3)
    _layer(lib, layers[0], rng, row_sample=64)


def test_llama3_8b_block_all_bits(lib):
    """The seven linears of the block, each X once; bits 2 (ternary), 3 and 4 across the
    linears. U is compared in full for the 4096-wide inputs; the 14336-wide input's U is
    the same computation the MLP-down test compares in full."""
    wl, layers = bench.build_layers(4, "cuda")
    rng = np.random.default_rng(4)
    # layers come per bit width as [q/k/v, o, gate/up, down]; inputs repeat across widths
    want = {0: 2, 1: 3, 2: 4, 3: 2}
    picked = [L for i, L in enumerate(layers) if L.spec.q.bits == want[i % 4]]
    assert len(picked) == 4
    for L in picked:
        _layer(lib, L, rng, row_sample=32, check_u=L.X.shape[1] <= 4096)
        torch.cuda.empty_cache()
