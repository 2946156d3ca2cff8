"""The layer-wise pipeline (GPTQ guide page, `apply_layerwise`) on the GPU against the
oracle.

Per layer, on the calibration input the GPU pipeline actually produced (bf16 outputs of
the already-quantised layers before it):
  H   relative Frobenius <= 1e-5 against the oracle's 2 h^T h / n from the same bf16 bits
  U   relative Frobenius <= 1e-4 against the oracle's inv + Cholesky of the GPU's H
  codes teacher-forced through the oracle loop given the GPU's U: >= 99.99% identical,
      mismatches only at half-points; packed words bit-exact
  forward  the next layer's input (bf16) against relu(h Wq^T) from the GPU's Wq, within
      bf16 rounding of the weights and of the output plus fp32 accumulation:
      |dy| <= 2^-9 |y| + (2^-9 + K 2^-23) sum_k |h_k||w_k|
End to end, the relative output error of the quantised network (against the float
network on the same input) is within 2% of the oracle pipeline's, which rounds its
activations to bf16 the same way.
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


def _run(lib, spec, seed):
    X = synth.make_x(spec.x, seed, device=DEV)
    Ws = synth.make_mlp_weights(spec, seed + 100, device=DEV)
    layers, out = lib.gptq_layerwise(X, Ws, spec.bits, spec.group, spec.sym, spec.damp, spec.act_order)
    torch.cuda.synchronize()
    return X, Ws, layers, out


CASES = [("toy", None), ("toy", dict(bits=4, group=64, sym=False, act_order=True))]


@pytest.mark.parametrize("name,over", CASES)
def test_layerwise_per_layer_parity(lib, name, over):
    spec = synth.mlp_workload(name)
    if over:
        import dataclasses
        spec = dataclasses.replace(spec, **over)
    X, Ws, layers, out = _run(lib, spec, 31)
    for i, L in enumerate(layers):
        h = synth.to_numpy_f64(L["input"])
        n = h.shape[0]
        S = O.xtx(h)
        Href = O.hessian_from_sum(S, n)
        Hg = npy(L["H"]).astype(np.float64)
        assert np.linalg.norm(Hg - Href) <= 1e-5 * np.linalg.norm(Href), i
        Uref, pref, dref = O.prepare(Hg, spec.damp, spec.act_order, np.diag(S))
        Ug = npy(L["U"]).astype(np.float64)
        assert np.linalg.norm(Ug - Uref) <= 1e-4 * np.linalg.norm(Uref), i
        W = synth.to_numpy_f64(Ws[i])
        codes = npy(L["codes"]).astype(np.int64)
        zeros = npy(L["zeros"]).astype(np.int64)
        forced = O.gptq_quantize(W, Ug, npy(L["perm"]), npy(L["dead"]).astype(bool), spec.bits, spec.group, spec.sym,
                                 forced_codes=codes, forced_zeros=None if spec.sym else zeros)
        nmis = len([t for t in forced["ties"] if t[2] == "code"])
        assert nmis <= 1e-4 * codes.size + 0.5, (i, forced["ties"][:3])
        np.testing.assert_array_equal(npy(L["packed"]).view(np.uint32), forced["packed"])
        # forward: the next layer's input from this layer's stored form
        Wq = npy(L["Wq"]).astype(np.float64)
        y = h @ Wq.T
        last = i == len(layers) - 1
        if not last:
            y = np.maximum(y, 0.0)
        got = synth.to_numpy_f64(layers[i + 1]["input"]) if not last else npy(out).astype(np.float64)
        K = h.shape[1]
        bound = (0.0 if last else 2.0 ** -9) * np.abs(y) + (2.0 ** -9 + K * 2.0 ** -23) * (np.abs(h) @ np.abs(Wq).T)
        assert np.all(np.abs(got - y) <= bound + 1e-30), i


@pytest.mark.parametrize("name,over", CASES)
def test_layerwise_output_error_matches_oracle_pipeline(lib, name, over):
    spec = synth.mlp_workload(name)
    if over:
        import dataclasses
        spec = dataclasses.replace(spec, **over)
    X, Ws, layers, out = _run(lib, spec, 41)
    Xh = synth.to_numpy_f64(X)
    Wh = [synth.to_numpy_f64(W) for W in Ws]
    ref = O.mlp_forward(Xh, Wh)
    err = lambda y: float(np.sum((y - ref) ** 2) / np.sum(ref ** 2))
    fn = lambda W, h: O.gptq_layer(W, h, spec.bits, spec.group, spec.sym, spec.damp, spec.act_order)["Wq"]
    _, _, y_ref = O.apply_layerwise(Xh, Wh, fn, act_round=O.round_bf16)
    e_gpu, e_ref = err(npy(out).astype(np.float64)), err(y_ref)
    print(f"{spec.name}: relative output error gpu {e_gpu:.6f} oracle {e_ref:.6f}")
    assert abs(e_gpu - e_ref) <= 0.02 * e_ref
    # and layer-wise GPTQ beats layer-wise RTN (the guide page's simulation claim)
    _, _, y_rtn = O.apply_layerwise(Xh, Wh, lambda W, h: O.rtn_quantize(W, spec.bits, spec.group, spec.sym)["Wq"],
                                    act_round=O.round_bf16)
    assert e_gpu < err(y_rtn)


def test_layerwise_mlp4096_sampled(lib):
    """The wide layer-wise case (three 4096-wide layers on 8192 tokens, 4-bit g128), with the
    per-layer checks on samples the oracle computes one by one: H in full (relative
    Frobenius 1e-5); U in full; codes teacher-forced on a sample of rows; the sampled rows'
    output error from the oracle's own fp64 H -> U chain within 2% of the GPU's; and the next
    layer's input on the sampled output columns (within bf16 rounding of weights and outputs).

    U's tolerance: 1e-4 relative where the equilibrated, damped Hessian is well conditioned
    (kappa <= 1e3, as on every benchmarked workload, kappa ~ 2-10). The hidden layers here
    see ReLU outputs on only n = 2d tokens, kappa ~ 2e5: there any fp32 factorization is only
    bound by the first-order forward error kappa * 2^-24 of a Cholesky factor, which is
    what is asserted (the output-error check carries the method-level claim)."""
    spec = synth.mlp_workload("mlp4096")
    X, Ws, layers, out = _run(lib, spec, 51)
    rng = np.random.default_rng(51)
    for i, L in enumerate(layers):
        h = synth.to_numpy_f64(L["input"])
        n = h.shape[0]
        S = O.xtx(h)
        Href = O.hessian_from_sum(S, n)
        Hg = npy(L["H"]).astype(np.float64)
        assert np.linalg.norm(Hg - Href) <= 1e-5 * np.linalg.norm(Href), i
        Hd = O.add_damping(O.fix_dead(Hg), spec.damp)
        dg = np.sqrt(np.diag(Hd))
        ev = np.linalg.eigvalsh(Hd / np.outer(dg, dg))
        kappa = ev[-1] / ev[0]
        Uref, pref, dref = O.prepare(Hg, spec.damp, spec.act_order, np.diag(S))
        Ug = npy(L["U"]).astype(np.float64)
        rel_u = np.linalg.norm(Ug - Uref) / np.linalg.norm(Uref)
        tol_u = 1e-4 if kappa <= 1e3 else kappa * 2.0 ** -24
        print(f"layer {i}: kappa {kappa:.3g}, U rel {rel_u:.3g} (tolerance {tol_u:.3g})")
        assert rel_u <= tol_u, (i, kappa, rel_u)
        del Uref
        rows = np.sort(rng.choice(Ws[i].shape[0], 24, replace=False))
        ri = torch.as_tensor(rows, device=DEV)
        W = synth.to_numpy_f64(Ws[i][ri])
        codes = npy(L["codes"][ri]).astype(np.int64)
        forced = O.gptq_quantize(W, Ug, npy(L["perm"]), npy(L["dead"]).astype(bool), spec.bits, spec.group,
                                 spec.sym, forced_codes=codes)
        nmis = len([t for t in forced["ties"] if t[2] == "code"])
        assert nmis <= 1e-4 * codes.size + 0.5, (i, forced["ties"][:3])
        np.testing.assert_array_equal(npy(L["packed"][ri]).view(np.uint32), forced["packed"])
        # the oracle's own chain from the same layer input: its fp64 H, its U, its free loop
        Uo, po, do = O.prepare(Href, spec.damp, spec.act_order, np.diag(S))
        free = O.gptq_quantize(W, Uo, po, do, spec.bits, spec.group, spec.sym)
        del Uo
        Wq = npy(L["Wq"][ri]).astype(np.float64)
        e_gpu = O.rel_output_error_from_xtx(S, W, Wq)
        e_ref = O.rel_output_error_from_xtx(S, W, free["Wq"])
        print(f"layer {i}: sampled rows' output error gpu {e_gpu:.6f} oracle chain {e_ref:.6f}")
        assert abs(e_gpu - e_ref) <= 0.02 * e_ref, (i, e_gpu, e_ref)
        # forward on the sampled output columns
        y = h @ Wq.T
        last = i == len(layers) - 1
        if not last:
            y = np.maximum(y, 0.0)
        nxt = layers[i + 1]["input"] if not last else out
        got = npy(nxt[:, ri].float()).astype(np.float64)
        K = h.shape[1]
        bound = (0.0 if last else 2.0 ** -9) * np.abs(y) + (2.0 ** -9 + K * 2.0 ** -23) * (np.abs(h) @ np.abs(Wq).T)
        assert np.all(np.abs(got - y) <= bound + 1e-30), i
