"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle, stage by stage.

Tolerances:
  H        relative Frobenius <= 1e-5 against fp64 H on the same bf16/fp32 bits
  U        relative Frobenius <= 1e-4, the GPU prepare fed the oracle's H rounded to fp32
  codes    given the oracle's U: >= 99.99% identical, every mismatch within 1e-4 (code
           units) of a rounding half-point, checked by the teacher-forced oracle
  RTN, packing, perm, dead, g_idx: bit-exact
  end to end: relative output error within 2% of the oracle's
"""
import numpy as np
import pytest
import torch

import oracle as O
import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"


def rel_fro(a, b):
    return float(np.linalg.norm(np.asarray(a, np.float64) - b) / np.linalg.norm(b))


def npy(t):
    return t.detach().cpu().numpy()


def f32(a):
    return np.ascontiguousarray(np.asarray(a, np.float64).astype(np.float32))


def x_case(n, d, seed, dead_frac=0.0, kind="scaled", dtype="bf16"):
    spec = synth.XSpec(n=n, d=d, kind=kind, dtype=dtype, n_outliers=max(1, d // 64), outlier_factor=20.0,
                       dead_frac=dead_frac, segment=1024)
    return synth.make_x(spec, seed, device=DEV)


# ------------------------------------------------------------------------------ Hessian

@pytest.mark.parametrize("n,d,dtype", [(512, 256, "f32"), (4096, 256, "bf16"), (8192, 768, "bf16"),
                                       (3000, 384, "bf16"), (1000, 200, "bf16"), (9000, 1024, "bf16"),
                                       (777, 136, "f32")])
def test_hessian_matches_oracle(lib, n, d, dtype):
    X = x_case(n, d, 10 + d, dead_frac=0.02, dtype=dtype)
    h = lib.Hessian(d)
    h.accumulate(X)
    H, diag, nn = h.finalize()
    Xh = synth.to_numpy_f64(X)
    S = O.xtx(Xh)
    Href = O.hessian_from_sum(S, n)
    assert nn == n
    assert rel_fro(npy(H), Href) <= 1e-5
    np.testing.assert_allclose(npy(diag), np.diag(S), rtol=2e-5, atol=0)
    Hg = npy(H)
    np.testing.assert_array_equal(Hg, Hg.T)                      # both triangles written
    dead = np.diag(Href) == 0
    assert np.all(np.diag(Hg)[dead] == 0)                        # dead channels stay exactly 0


def test_hessian_streaming_equals_one_call(lib):
    d = 512
    X = x_case(6000, d, 77)
    a = lib.Hessian(d)
    a.accumulate(X)
    Ha, _, _ = a.finalize()
    b = lib.Hessian(d)
    for r in range(0, 6000, 2048):
        b.accumulate(X[r:r + 2048])
    Hb, _, n = b.finalize()
    assert n == 6000
    Href = O.hessian(synth.to_numpy_f64(X))
    assert rel_fro(npy(Hb), Href) <= 1e-5
    assert rel_fro(npy(Ha), npy(Hb).astype(np.float64)) <= 1e-5
    b.reset()
    b.accumulate(X[:100])
    Hc, _, n = b.finalize()
    assert n == 100 and rel_fro(npy(Hc), O.hessian(synth.to_numpy_f64(X[:100]))) <= 1e-5


def test_hessian_bf16_unaligned_rows_use_simt_path(lib):
    d = 200
    base = x_case(1500, d + 1, 5)
    X = base[:, :d]                                              # row stride 201 elements: not TMA-addressable
    h = lib.Hessian(d)
    h.accumulate(X)
    H, _, _ = h.finalize()
    assert rel_fro(npy(H), O.hessian(synth.to_numpy_f64(X))) <= 1e-5


# ------------------------------------------------------------------------------ prepare

def _h_for(d, seed, dead_frac=0.02, n=None):
    X = x_case(n or 4 * d, d, seed, dead_frac=dead_frac)
    Xh = synth.to_numpy_f64(X)
    S = O.xtx(Xh)
    H32 = f32(O.hessian_from_sum(S, Xh.shape[0]))
    return H32, f32(np.diag(S)), Xh


@pytest.mark.parametrize("d,act_order", [(256, False), (768, False), (300, True), (1000, True), (129, False),
                                         (2048, True), (2100, False), (2176, True)])
def test_prepare_matches_oracle(lib, d, act_order):
    H32, diag32, _ = _h_for(d, 100 + d)
    U, perm, dead = lib.gptq_prepare(torch.tensor(H32, device=DEV), torch.tensor(diag32, device=DEV), 0.01,
                                     act_order=act_order)
    Uref, pref, dref = O.prepare(H32.astype(np.float64), 0.01, act_order, diag32.astype(np.float64))
    np.testing.assert_array_equal(npy(perm), pref)
    np.testing.assert_array_equal(npy(dead).astype(bool), dref)
    Ug = npy(U)
    assert np.all(np.tril(Ug, -1) == 0)
    assert np.all(np.diag(Ug) > 0)
    assert rel_fro(Ug, Uref) <= 1e-4


def test_prepare_reports_not_spd(lib):
    H = torch.tensor([[1.0, 2.0], [2.0, 1.0]], device=DEV)
    with pytest.raises(lib.GptqError) as e:
        lib.gptq_prepare(H, None, 0.0)
    assert e.value.status == 3


# ----------------------------------------------------------------------------- quantize

QCASES = [
    # rows, cols, bits, group, sym, act_order
    (128, 256, 4, 0, True, False),
    (96, 384, 4, 128, False, False),
    (64, 300, 3, 32, True, True),
    (48, 512, 2, 256, True, False),
    (33, 200, 4, 64, False, True),
    (130, 640, 3, 128, True, True),
    (40, 384, 2, 128, False, False),
    # asymmetric 2- and 3-bit with act_order (the paper's default grid, narrow widths)
    (72, 256, 2, 128, False, True),
    (50, 384, 3, 32, False, True),
    # several super-blocks of the deferred trailing update, ragged last block
    (64, 1100, 4, 128, False, True),
    # cols % 4 != 0: the FFMA trailing update (TMA needs 16-byte rows) and the any-length packer
    (130, 301, 4, 128, False, True),
    (70, 458, 3, 0, True, False),
]


@pytest.mark.parametrize("rows,cols,bits,group,sym,act", QCASES)
def test_quantize_given_oracle_u(lib, rows, cols, bits, group, sym, act):
    H32, diag32, _ = _h_for(cols, 200 + cols + rows)
    Uref, perm, dead = O.prepare(H32.astype(np.float64), 0.01, act, diag32.astype(np.float64))
    U32 = f32(Uref)
    W = synth.make_weight(rows, cols, 0.02, 300 + rows, device=DEV)
    Wh = synth.to_numpy_f64(W)
    out = lib.gptq_quantize(W, torch.tensor(U32, device=DEV), torch.tensor(perm.astype(np.int32), device=DEV),
                            torch.tensor(dead.astype(np.uint8), device=DEV), bits, group, sym)
    codes = npy(out["codes"]).astype(np.int64)
    zeros = npy(out["zeros"]).astype(np.int64)
    ref = O.gptq_quantize(Wh, U32.astype(np.float64), perm, dead, bits, group, sym, forced_codes=codes,
                          forced_zeros=None if sym else zeros)
    nmis = len([t for t in ref["ties"] if t[2] == "code"])
    assert nmis <= 1e-4 * codes.size + 0.5, ref["ties"]
    np.testing.assert_array_equal(codes, ref["codes"])
    np.testing.assert_allclose(npy(out["scales"]), ref["scales"], rtol=2e-5, atol=0)
    np.testing.assert_array_equal(zeros, ref["zeros"])
    np.testing.assert_allclose(npy(out["Wq"]), ref["Wq"], rtol=2e-5, atol=1e-7)
    np.testing.assert_array_equal(npy(out["g_idx"]), ref["g_idx"])
    np.testing.assert_array_equal(npy(out["packed"]).view(np.uint32), ref["packed"])
    np.testing.assert_allclose(npy(out["row_loss"]), ref["err_sq"], rtol=1e-3)
    assert np.all(npy(out["Wq"])[:, dead] == 0)


# ---------------------------------------------------------------------------------- RTN

@pytest.mark.parametrize("rows,cols,bits,group,sym", [(64, 256, 4, 0, True), (64, 256, 4, 128, False),
                                                      (37, 300, 3, 64, True), (16, 1000, 2, 128, True),
                                                      (9, 77, 3, 0, False)])
def test_rtn_bit_exact(lib, rows, cols, bits, group, sym):
    W = synth.make_weight(rows, cols, 0.05, 400 + cols, device=DEV)
    dead = torch.zeros(cols, dtype=torch.uint8, device=DEV)
    dead[::17] = 1
    out = lib.rtn_quantize(W, bits, group, sym, dead=dead)
    ref = O.rtn_quantize(synth.to_numpy_f64(W), bits, group, sym, dead=npy(dead).astype(bool))
    np.testing.assert_array_equal(npy(out["codes"]).astype(np.int64), ref["codes"])
    np.testing.assert_array_equal(npy(out["scales"]), f32(ref["scales"]))
    np.testing.assert_array_equal(npy(out["zeros"]).astype(np.int64), ref["zeros"])
    np.testing.assert_array_equal(npy(out["Wq"]), f32(ref["Wq"]))
    np.testing.assert_array_equal(npy(out["packed"]).view(np.uint32), ref["packed"])


# asymmetric grid over the range widened to contain 0: rows shifted so most groups are
# one-signed (where the widening changes the grid)
ZCASES = [(64, 256, 4, 128, False), (50, 384, 3, 32, True), (40, 300, 2, 0, True), (33, 640, 3, 128, True)]


@pytest.mark.parametrize("rows,cols,bits,group,act", ZCASES)
def test_quantize_zero_in_range_given_oracle_u(lib, rows, cols, bits, group, act):
    # no dead inputs here: a zeroed dead column puts 0 into its group's range by itself
    H32, diag32, _ = _h_for(cols, 500 + cols + rows, dead_frac=0.0)
    Uref, perm, dead = O.prepare(H32.astype(np.float64), 0.01, act, diag32.astype(np.float64))
    U32 = f32(Uref)
    W = synth.make_weight(rows, cols, 0.02, 600 + rows, device=DEV)
    W += torch.linspace(-0.1, 0.1, rows, device=DEV)[:, None]
    Wh = synth.to_numpy_f64(W)
    out = lib.gptq_quantize(W, torch.tensor(U32, device=DEV), torch.tensor(perm.astype(np.int32), device=DEV),
                            torch.tensor(dead.astype(np.uint8), device=DEV), bits, group, False, zero_in_range=True)
    codes = npy(out["codes"]).astype(np.int64)
    zeros = npy(out["zeros"]).astype(np.int64)
    ref = O.gptq_quantize(Wh, U32.astype(np.float64), perm, dead, bits, group, False, forced_codes=codes,
                          forced_zeros=zeros, zero_in_range=True)
    nmis = len([t for t in ref["ties"] if t[2] == "code"])
    assert nmis <= 1e-4 * codes.size + 0.5, ref["ties"]
    np.testing.assert_array_equal(codes, ref["codes"])
    np.testing.assert_allclose(npy(out["scales"]), ref["scales"], rtol=2e-5, atol=0)
    np.testing.assert_array_equal(zeros, ref["zeros"])
    np.testing.assert_allclose(npy(out["Wq"]), ref["Wq"], rtol=2e-5, atol=1e-7)
    np.testing.assert_array_equal(npy(out["g_idx"]), ref["g_idx"])
    np.testing.assert_array_equal(npy(out["packed"]).view(np.uint32), ref["packed"])
    # the widened grid differs from the raw one on these rows (one-signed groups get
    # another scale), and 0 is a grid point of every group: code z dequantises to 0
    raw = O.gptq_quantize(Wh, U32.astype(np.float64), perm, dead, bits, group, False)
    assert np.mean(raw["scales"] != ref["scales"]) > 0.2


@pytest.mark.parametrize("rows,cols,bits,group", [(64, 256, 4, 128), (37, 300, 3, 64), (16, 1000, 2, 128),
                                                  (9, 77, 3, 0)])
def test_rtn_zero_in_range_bit_exact(lib, rows, cols, bits, group):
    W = synth.make_weight(rows, cols, 0.05, 700 + cols, device=DEV)
    W += torch.linspace(-0.2, 0.2, rows, device=DEV)[:, None]
    dead = torch.zeros(cols, dtype=torch.uint8, device=DEV)
    dead[::17] = 1
    out = lib.rtn_quantize(W, bits, group, False, dead=dead, zero_in_range=True)
    ref = O.rtn_quantize(synth.to_numpy_f64(W), bits, group, False, dead=npy(dead).astype(bool), zero_in_range=True)
    np.testing.assert_array_equal(npy(out["codes"]).astype(np.int64), ref["codes"])
    np.testing.assert_array_equal(npy(out["scales"]), f32(ref["scales"]))
    np.testing.assert_array_equal(npy(out["zeros"]).astype(np.int64), ref["zeros"])
    np.testing.assert_array_equal(npy(out["Wq"]), f32(ref["Wq"]))
    np.testing.assert_array_equal(npy(out["packed"]).view(np.uint32), ref["packed"])


def _tie_segment(rng, n, bits, sym):
    """n fp32 weights whose grid (from their own min/max) puts many of them exactly on, or
    one ulp either side of, a rounding half-point of w / s (+ z)."""
    f = np.float32
    if sym:
        qm = 2 ** (bits - 1) - 1
        mx = f(rng.uniform(0.05, 0.5))
        s = f(np.float64(mx) / qm)
        z = 0
        lo_w, hi_w = -mx, mx
        ks = np.arange(-qm, qm)
    else:
        qm = 2 ** bits - 1
        mn, mx = f(-rng.uniform(0.05, 0.5)), f(rng.uniform(0.05, 0.5))
        s = f((np.float64(mx) - np.float64(mn)) / qm)
        z = int(min(max(np.rint(-np.float64(mn) / np.float64(s)), 0), qm))
        lo_w, hi_w = mn, mx
        ks = np.arange(0, qm)
    vals = [hi_w, lo_w]
    for k in ks:
        t = f((k + 0.5 - z) * np.float64(s))
        for v in (t, np.nextafter(t, f(np.inf)), np.nextafter(t, f(-np.inf))):
            if lo_w <= v <= hi_w:
                vals.append(f(v))
    vals = np.array(vals, dtype=f)
    out = rng.choice(vals[2:], n)
    out[:2] = vals[:2]
    return out


@pytest.mark.parametrize("bits,group,sym", [(4, 0, True), (3, 0, False), (4, 32, False), (2, 64, True)])
def test_rtn_exact_at_half_points(lib, bits, group, sym):
    """Weights on and one ulp around the half-points of their own grid: the codes must be
    the exact round-half-even decisions (bit-exact against the fp64 oracle)."""
    rng = np.random.default_rng(bits * 10 + group)
    rows, cols = 24, 128
    step = group if group else cols
    W = np.concatenate([np.stack([_tie_segment(rng, step, bits, sym) for _ in range(rows)])
                        for _ in range(cols // step)], axis=1)
    Wt = torch.tensor(W, device=DEV)
    out = lib.rtn_quantize(Wt, bits, group, sym)
    ref = O.rtn_quantize(W.astype(np.float64), bits, group, sym)
    np.testing.assert_array_equal(npy(out["scales"]), f32(ref["scales"]))
    np.testing.assert_array_equal(npy(out["codes"]).astype(np.int64), ref["codes"])


@pytest.mark.parametrize("bits,sym,cols,rows", [(2, True, 64, 11), (3, True, 96, 11), (3, False, 100, 11),
                                                (4, False, 33, 11), (4, True, 4096, 301), (3, True, 3072, 97),
                                                (2, False, 1024, 257), (4, False, 14336, 5)])
def test_pack_bit_exact(lib, bits, sym, cols, rows):
    """Rows of a multiple of 32 codes take the 32-codes-per-thread packer, others the
    one-word-per-thread packer; both bit-exact against the oracle's bitstream."""
    rng = np.random.default_rng(bits * 100 + cols)
    lo, hi = (-(2 ** (bits - 1) - 1), 2 ** (bits - 1) - 1) if sym else (0, 2 ** bits - 1)
    codes = rng.integers(lo, hi + 1, size=(rows, cols))
    p = lib.gptq_pack(torch.tensor(codes.astype(np.int8), device=DEV), bits, sym)
    np.testing.assert_array_equal(npy(p).view(np.uint32), O.pack_rows(O.unsigned_codes(codes, bits, sym), bits))


def test_pack_misaligned_codes_take_the_general_packer(lib):
    """Codes that do not start on a 16-byte boundary (a view one byte into a buffer) are packed
    by the general kernel, with the same result."""
    rng = np.random.default_rng(5)
    codes = rng.integers(-7, 8, size=(40, 256)).astype(np.int8)
    buf = torch.zeros(codes.size + 1, dtype=torch.int8, device=DEV)
    buf[1:] = torch.tensor(codes.reshape(-1), device=DEV)
    view = buf[1:].view(40, 256)
    assert view.data_ptr() % 16 != 0
    p = lib.gptq_pack(view, 4, True)
    np.testing.assert_array_equal(npy(p).view(np.uint32), O.pack_rows(O.unsigned_codes(codes, 4, True), 4))


# ---------------------------------------------------------------------------- end to end

def _layer_gpu(lib, X, Ws, bits, group, sym, act_order, damp=0.01):
    h = lib.Hessian(X.shape[1])
    h.accumulate(X)
    H, diag, _ = h.finalize()
    U, perm, dead = lib.gptq_prepare(H, diag, damp, act_order=act_order)
    outs = [lib.gptq_quantize(W, U, perm, dead, bits, group, sym) for W in Ws]
    return outs, (H, U, perm, dead)


@pytest.mark.parametrize("cfg", [0, 1])
def test_end_to_end_output_error(lib, cfg):
    wl = synth.workload(cfg)
    L = wl.layers[0]
    X = synth.make_x(L.x, synth.x_seed(cfg, L.x), device=DEV)
    Ws = [synth.make_weight(w.out, w.inp, w.std, synth.weight_seed(cfg, w.name), device=DEV) for w in L.weights]
    outs, (H, U, perm, dead) = _layer_gpu(lib, X, Ws, L.q.bits, L.q.group, L.q.sym, L.q.act_order)
    Xh = synth.to_numpy_f64(X)
    S = O.xtx(Xh)
    for W, out in zip(Ws, outs):
        Wh = synth.to_numpy_f64(W)
        ref = O.gptq_layer(Wh, Xh, L.q.bits, L.q.group, L.q.sym, L.q.damp, L.q.act_order)
        e_gpu = O.rel_output_error_from_xtx(S, Wh, npy(out["Wq"]))
        e_ref = O.rel_output_error_from_xtx(S, Wh, ref["Wq"])
        assert abs(e_gpu - e_ref) <= 0.02 * e_ref, (e_gpu, e_ref)
        rtn = lib.rtn_quantize(W, L.q.bits, L.q.group, L.q.sym, dead=dead)
        e_rtn = O.rel_output_error_from_xtx(S, Wh, npy(rtn["Wq"]))
        assert e_gpu < e_rtn, (e_gpu, e_rtn)
        np.testing.assert_array_equal(npy(dead).astype(bool), ref["dead"])


@pytest.mark.parametrize("group,sym", [(0, True), (64, True), (128, False)])
def test_diagonal_hessian_gives_rtn_on_gpu(lib, group, sym):
    """X = Hadamard columns: H = 2I exactly in fp32, U diagonal, GPTQ == RTN bit for bit."""
    spec = synth.XSpec(n=512, d=256, kind="hadamard", dtype="bf16")
    X = synth.make_x(spec, 0, device=DEV)
    W = synth.make_weight(128, 256, 0.1, 7, device=DEV)
    outs, (H, U, perm, dead) = _layer_gpu(lib, X, [W], 4, group, sym, False)
    assert torch.equal(H, 2 * torch.eye(256, device=DEV))
    Ug = npy(U)
    assert np.count_nonzero(Ug - np.diag(np.diag(Ug))) == 0
    r = lib.rtn_quantize(W, 4, group, sym)
    assert torch.equal(outs[0]["codes"], r["codes"])
    assert torch.equal(outs[0]["packed"], r["packed"])


@pytest.mark.parametrize("bits,group,sym,act", [(4, 128, True, False), (3, 128, False, True), (2, 0, True, False)])
def test_correlated_channels_gptq_beats_rtn(lib, bits, group, sym, act):
    """Correlated channels (X = Z A): a Hessian far from diagonal, where GPTQ's error
    compensation has room to work; the GPU's output error is within 2% of the oracle's
    and below round-to-nearest's."""
    spec = synth.XSpec(n=8192, d=1024, kind="correlated", dtype="bf16", segment=2048)
    X = synth.make_x(spec, 31 + bits, device=DEV)
    W = synth.make_weight(512, 1024, 0.02, 41 + bits, device=DEV)
    outs, (H, U, perm, dead) = _layer_gpu(lib, X, [W], bits, group, sym, act)
    Xh = synth.to_numpy_f64(X)
    Wh = synth.to_numpy_f64(W)
    S = O.xtx(Xh)
    ref = O.gptq_layer(Wh, Xh, bits, group, sym, 0.01, act)
    e_gpu = O.rel_output_error_from_xtx(S, Wh, npy(outs[0]["Wq"]))
    e_ref = O.rel_output_error_from_xtx(S, Wh, ref["Wq"])
    rtn = lib.rtn_quantize(W, bits, group, sym, dead=dead)
    e_rtn = O.rel_output_error_from_xtx(S, Wh, npy(rtn["Wq"]))
    assert abs(e_gpu - e_ref) <= 0.02 * e_ref, (e_gpu, e_ref)
    assert e_gpu < 0.9 * e_rtn, (e_gpu, e_rtn)


def test_stacked_weights_equal_per_weight_calls(lib):
    """Rows are independent given U: one gptq_quantize over the weights of a layer stacked
    by rows gives, row for row, exactly what one call per weight gives. (The benchmark
    quantises each layer's weights stacked, as one fused projection.)"""
    import bench
    wl, layers = bench.build_layers(1, DEV)
    L = layers[0]
    q = L.spec.q
    h = lib.Hessian(L.X.shape[1])
    h.accumulate(L.X)
    H, diag, _ = h.finalize()
    U, perm, dead = lib.gptq_prepare(H, diag, q.damp, act_order=q.act_order)
    cat = lib.gptq_quantize(L.Wcat, U, perm, dead, q.bits, q.group, q.sym)
    r0 = 0
    for W in L.Ws:
        one = lib.gptq_quantize(W, U, perm, dead, q.bits, q.group, q.sym)
        r1 = r0 + W.shape[0]
        for k in ("codes", "scales", "zeros", "Wq", "packed", "row_loss"):
            assert torch.equal(cat[k][r0:r1], one[k]), k
        assert torch.equal(cat["g_idx"], one["g_idx"])
        r0 = r1
    # the benchmark's runner: one step, outputs split back per weight
    runner = bench.Runner(lib, layers, torch.device(DEV))
    runner.step()
    torch.cuda.synchronize()
    parts = runner.weight_outputs(0)
    assert [p["codes"].shape[0] for p in parts] == [W.shape[0] for W in L.Ws]
    assert all(bool(torch.isfinite(p["Wq"]).all()) for p in parts)


def test_prepare_on_concurrent_streams_equals_sequential(lib):
    """gptq_prepare calls on different caller streams get their own library stream sets and
    run side by side on the GPU; each gives the result it gives alone, bit for bit (two
    super-panel sizes and one small one, all three in flight at once)."""
    cases = [(2176, True, 601), (2304, False, 602), (768, False, 603)]
    inputs = []
    for d, act, seed in cases:
        H32, diag32, _ = _h_for(d, seed)
        inputs.append((torch.tensor(H32, device=DEV), torch.tensor(diag32, device=DEV), act,
                       torch.empty(lib.gptq_prepare_workspace_bytes(d, True), dtype=torch.uint8, device=DEV)))
    ref = []
    for H, diag, act, ws in inputs:
        U, perm, dead = lib.gptq_prepare(H, diag, 0.01, act_order=act, ws=ws)
        torch.cuda.synchronize()
        ref.append((npy(U), npy(perm), npy(dead)))
    streams = [torch.cuda.Stream() for _ in inputs]
    outs = []
    with lib.deferred_status():
        for st, (H, diag, act, ws) in zip(streams, inputs):
            st.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(st):
                outs.append(lib.gptq_prepare(H, diag, 0.01, act_order=act, ws=ws))
        for st in streams:
            torch.cuda.current_stream().wait_stream(st)
        lib.status_sync()
    torch.cuda.synchronize()
    for (U, perm, dead), (Ur, pr, dr) in zip(outs, ref):
        np.testing.assert_array_equal(npy(U), Ur)
        np.testing.assert_array_equal(npy(perm), pr)
        np.testing.assert_array_equal(npy(dead), dr)


def test_prepare_on_more_caller_streams_than_sets(lib):
    """Eleven gptq_prepare calls in flight on eleven caller streams (more than the 8 stream
    sets per device, so some calls share a set and take its streams in turn; three of the
    callers are high-priority streams, whose factorisations' side streams take that
    priority): each gives its sequential result bit for bit."""
    sizes = [256, 384, 512, 640, 768, 256, 384, 512, 640, 768, 2176]
    inputs = []
    for i, d in enumerate(sizes):
        H32, diag32, _ = _h_for(d, 700 + i)
        inputs.append((torch.tensor(H32, device=DEV), torch.tensor(diag32, device=DEV), i % 2 == 0,
                       torch.empty(lib.gptq_prepare_workspace_bytes(d, True), dtype=torch.uint8, device=DEV)))
    ref = []
    for H, diag, act, ws in inputs:
        U, perm, dead = lib.gptq_prepare(H, diag, 0.01, act_order=act, ws=ws)
        torch.cuda.synchronize()
        ref.append((npy(U), npy(perm), npy(dead)))
    streams = [torch.cuda.Stream(priority=-1 if i % 4 == 1 else 0) for i in range(len(inputs))]
    outs = []
    with lib.deferred_status():
        for st, (H, diag, act, ws) in zip(streams, inputs):
            st.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(st):
                outs.append(lib.gptq_prepare(H, diag, 0.01, act_order=act, ws=ws))
        for st in streams:
            torch.cuda.current_stream().wait_stream(st)
        lib.status_sync()
    torch.cuda.synchronize()
    for (U, perm, dead), (Ur, pr, dr) in zip(outs, ref):
        np.testing.assert_array_equal(npy(U), Ur)
        np.testing.assert_array_equal(npy(perm), pr)
        np.testing.assert_array_equal(npy(dead), dr)
