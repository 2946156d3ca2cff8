"""Pins for the CPU oracle: facts that do not come from the oracle itself.

Each test checks the oracle against something the pages or the mathematics fix —
hand-computed values, closed forms, brute-force OBS, limit cases that reduce to
round-to-nearest, and the seeded demo printed on the AutoGPTQ page — chosen so
that a dropped term, a wrong sign or index, or a transposed operand in the
oracle fails at least one of them.
"""
import json
import os

import numpy as np
import pytest

import oracle as O
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _damped(H, damp=0.01):
    return O.add_damping(O.fix_dead(H), damp)


# -------------------------------------------------------------------------- Hessian

def test_hessian_by_hand():
    # X^T X for X = [[1,2],[3,4],[0,1]] is [[10,14],[14,21]]; n = 3.
    X = np.array([[1.0, 2.0], [3.0, 4.0], [0.0, 1.0]])
    H = O.hessian(X)
    np.testing.assert_array_equal(H * 3 / 2, np.array([[10.0, 14.0], [14.0, 21.0]]))


def test_hessian_streaming_equals_one_shot():
    X = _rng(1).standard_normal((300, 7))
    S, n = O.hessian_accumulate([X[:128], X[128:256], X[256:]])
    assert n == 300
    np.testing.assert_allclose(O.hessian_from_sum(S, n), O.hessian(X), rtol=1e-13, atol=1e-14)


def test_dead_fix_and_damping_by_hand():
    H = np.array([[4.0, 1.0, 0.0], [1.0, 3.0, 0.0], [0.0, 0.0, 0.0]])
    np.testing.assert_array_equal(O.dead_mask(H), [False, False, True])
    Hf = O.fix_dead(H)
    np.testing.assert_array_equal(Hf, [[4, 1, 0], [1, 3, 0], [0, 0, 1]])
    Hd = O.add_damping(Hf, 0.03)          # mean diag after the fix = 8/3 -> +0.08
    np.testing.assert_allclose(np.diag(Hd), [4.08, 3.08, 1.08], rtol=0, atol=1e-15)
    assert Hd[0, 1] == 1.0 and Hd[1, 0] == 1.0


def test_upper_cholesky_of_inverse_2x2_closed_form():
    a, b, c = 5.0, 2.0, 3.0
    det = a * c - b * b
    u11 = np.sqrt(c / det)
    u12 = -b / (det * u11)
    u22 = np.sqrt(a / det - u12 ** 2)
    U = O.upper_cholesky_of_inverse(np.array([[a, b], [b, c]]))
    np.testing.assert_allclose(U, [[u11, u12], [0.0, u22]], rtol=1e-14, atol=1e-15)


def test_u_rows_are_eliminated_inverse_rows():
    # Trick 2: row j of U is row j of H_F^-1 (F = {j..d-1}) over sqrt(H_F^-1[j, j]),
    # with H_F^-1 from successive Gaussian elimination of H^-1.
    d = 6
    A = _rng(2).standard_normal((40, d))
    H = _damped(O.hessian(A))
    U = O.upper_cholesky_of_inverse(H)
    Hinv = np.linalg.inv(H)
    for j in range(d):
        row = Hinv[j, j:] / np.sqrt(Hinv[j, j])
        np.testing.assert_allclose(U[j, j:], row, rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(U[j, :j], 0.0, atol=0)
        Hinv = Hinv - np.outer(Hinv[:, j], Hinv[j, :]) / Hinv[j, j]
    # and the factorisation itself: U^T U H = I, positive diagonal
    U = O.upper_cholesky_of_inverse(H)
    np.testing.assert_allclose(U.T @ U @ H, np.eye(d), atol=1e-12)
    assert np.all(np.diag(U) > 0)


# ----------------------------------------------------------------------- quantizers

def test_qmax():
    assert [O.qmax_sym(b) for b in (2, 3, 4)] == [1, 3, 7]
    assert [O.maxq_asym(b) for b in (2, 3, 4)] == [3, 7, 15]


def test_sym_quantizer_by_hand_half_to_even_and_clip():
    # row max 0.875, qmax 7 -> scale 0.125 (exact in fp32); t = w / 0.125
    w = np.array([[0.875, -0.3125, 0.1875, 0.4375, 0.0625, 1.0]])
    s, z = O.sym_params(w[:, :5], 7)
    assert s[0] == 0.125 and z[0] == 0
    c = O.quant_codes(w, s[:, None], z[:, None], 4, True)
    # 7, -2.5 -> -2, 1.5 -> 2, 3.5 -> 4, 0.5 -> 0, 8 -> clipped to 7
    np.testing.assert_array_equal(c, [[7, -2, 2, 4, 0, 7]])
    np.testing.assert_array_equal(O.dequant(c, s[:, None], 0, True), [[0.875, -0.25, 0.25, 0.5, 0.0, 0.875]])


def test_sym_scale_floor_for_zero_row():
    s, _ = O.sym_params(np.zeros((1, 4)), 7, scale_dtype=None)
    assert s[0] == 1e-12 / 7


def test_asym_quantizer_by_hand():
    # 2 bits: maxq 3; min -0.5, max 1.0 -> scale 0.5, zero round(1.0) = 1
    b = np.array([[-0.5, 1.0, 0.25, 0.0]])
    s, z = O.asym_params(b, 3)
    assert s[0] == 0.5 and z[0] == 1
    c = O.quant_codes(b, s[:, None], z[:, None], 2, False)
    np.testing.assert_array_equal(c, [[0, 3, 2, 1]])          # round(1.5) = 2 (half to even)
    np.testing.assert_array_equal(O.dequant(c, s[:, None], z[:, None], False), [[-0.5, 1.0, 0.5, 0.0]])
    # all-positive block: -min/scale < 0, zero clamped to 0
    s2, z2 = O.asym_params(np.array([[0.5, 1.0]]), 3)
    assert z2[0] == 0 and np.isclose(s2[0], 0.5 / 3, rtol=1e-7)
    # constant block: scale 1.0
    s3, z3 = O.asym_params(np.array([[0.25, 0.25]]), 15)
    assert s3[0] == 1.0 and z3[0] == 0


def test_asym_zero_in_range_by_hand():
    """The variant whose range is widened to contain 0 (values worked by hand)."""
    # all-positive block, 2 bits: range [0, 1] -> scale 1/3, zero 0 (the raw range [0.5, 1]
    # would give scale 1/6 and no grid point at 0)
    s, z = O.asym_params(np.array([[0.5, 1.0]]), 3, scale_dtype=None, zero_in_range=True)
    assert np.isclose(s[0], 1.0 / 3.0, rtol=1e-15) and z[0] == 0
    c = O.quant_codes(np.array([[0.5, 1.0, 0.0]]), s[:, None], z[:, None], 2, False)
    np.testing.assert_array_equal(c, [[2, 3, 0]])            # 0.5 * 3 = 1.5 -> 2 (half to even)
    # all-negative block, 3 bits: range [-1.4, 0] -> scale 0.2, zero round(7) = 7 = maxq
    s, z = O.asym_params(np.array([[-1.4, -0.2]]), 7, scale_dtype=None, zero_in_range=True)
    assert np.isclose(s[0], 0.2, rtol=1e-15) and z[0] == 7
    c = O.quant_codes(np.array([[-1.4, -0.2, 0.0]]), s[:, None], z[:, None], 3, False)
    np.testing.assert_array_equal(c, [[0, 6, 7]])
    np.testing.assert_allclose(O.dequant(c, s[:, None], z[:, None], False), [[-1.4, -0.2, 0.0]], atol=1e-15)
    # a block that already straddles 0 is unchanged by the widening
    b = _rng(5).standard_normal((6, 16))
    b[:, 0], b[:, 1] = -1.0, 1.0
    for bits in (2, 3, 4):
        s1, z1 = O.asym_params(b, 2 ** bits - 1)
        s2, z2 = O.asym_params(b, 2 ** bits - 1, zero_in_range=True)
        np.testing.assert_array_equal(s1, s2)
        np.testing.assert_array_equal(z1, z2)


def test_asym_zero_in_range_zero_is_exact():
    """With the widened range every block has 0 on its grid: w = 0 quantises to code z,
    which dequantises to exactly 0, and z lies in [0, maxq] without clamping."""
    rng = _rng(6)
    for bits in (2, 3, 4):
        maxq = 2 ** bits - 1
        b = rng.standard_normal((200, 8)) * 0.1 + rng.choice([-0.3, 0.0, 0.3], size=(200, 1))
        s, z = O.asym_params(b, maxq, zero_in_range=True)
        mn, mx = np.minimum(b.min(1), 0), np.maximum(b.max(1), 0)
        assert np.all((-mn / s >= -0.5) & (-mn / s <= maxq + 0.5))   # no clamping needed
        c = O.quant_codes(np.zeros((200, 1)), s[:, None], z[:, None], bits, False)
        np.testing.assert_array_equal(c[:, 0], z)
        assert np.all(O.dequant(c, s[:, None], z[:, None], False) == 0.0)


def test_stored_scale_is_float32_grid():
    w = _rng(3).standard_normal((5, 9))
    s, _ = O.sym_params(w, 7)
    assert np.all(s.astype(np.float32).astype(np.float64) == s)


# ----------------------------------------------------------------------------- pack

def test_pack_4bit_by_hand():
    u = np.array([[1, 2, 3, 4, 5, 6, 7, 8]])
    np.testing.assert_array_equal(O.pack_rows(u, 4), np.array([[0x87654321]], dtype=np.uint32))


def test_pack_2bit_by_hand():
    u = np.zeros((1, 16), dtype=np.int64)
    u[0, :3] = [1, 2, 3]                   # 1 + (2 << 2) + (3 << 4) = 57
    np.testing.assert_array_equal(O.pack_rows(u, 2), [[57]])


def test_pack_3bit_straddles_words():
    u = np.full((1, 32), 7)
    np.testing.assert_array_equal(O.pack_rows(u, 3), [[0xFFFFFFFF] * 3])
    u[0, 10] = 5                           # bits 30, 31, 32 = 1, 0, 1
    np.testing.assert_array_equal(O.pack_rows(u, 3), [[0x7FFFFFFF, 0xFFFFFFFF, 0xFFFFFFFF]])


def test_pack_ragged_row_pads_zero_bits():
    u = np.full((2, 5), 3)
    w = O.pack_rows(u, 3)                  # 15 bits -> one word
    np.testing.assert_array_equal(w, [[0b011011011011011] * 1] * 2)


def test_g_idx_by_hand():
    np.testing.assert_array_equal(O.g_idx_for(np.array([2, 0, 3, 1]), 2, 4), [0, 1, 0, 1])
    np.testing.assert_array_equal(O.g_idx_for(None, 2, 5), [0, 0, 1, 1, 2])
    np.testing.assert_array_equal(O.g_idx_for(None, 0, 3), [0, 0, 0])


def test_act_order_perm_stable_descending():
    np.testing.assert_array_equal(O.act_order_perm([3.0, 1.0, 3.0, 0.0, 2.0]), [0, 2, 4, 1, 3])


# ------------------------------------------------------------------- the GPTQ loop

@pytest.mark.parametrize("d,group,sym,bits,zr", [(4, 0, True, 3, False), (6, 0, True, 2, False),
                                                 (8, 0, True, 4, False), (8, 4, True, 3, False),
                                                 (8, 4, False, 4, False), (6, 3, False, 2, False),
                                                 (8, 4, False, 3, True), (6, 0, False, 2, True)])
def test_cholesky_loop_equals_bruteforce_obs(d, group, sym, bits, zr):
    """P-1/P-2: the Cholesky-form loop equals explicit OBS with Gaussian elimination,
    and each step raises the loss by err_j^2 / 2 = e^2 / (2 Hinv_F[j, j])."""
    rng = _rng(10 + d + group)
    X = rng.standard_normal((3 * d, d)) @ rng.standard_normal((d, d))
    W = rng.standard_normal((5, d)) * 0.3
    H = _damped(O.hessian(X))
    U = O.upper_cholesky_of_inverse(H)
    if zr:
        W = W + 0.4   # mostly one-signed rows, where the widened range differs
    r = O.gptq_loop(W, U, bits, group, sym, zero_in_range=zr)
    for i in range(W.shape[0]):
        q, incr = O.obs_bruteforce_row(W[i], H, bits, group, sym, zero_in_range=zr)
        np.testing.assert_allclose(r["Q"][i], q, rtol=0, atol=1e-12)
    # error increments: OBS's e^2 / (2 Hinv_F[j, j]) summed over the steps equals the
    # loop's sum of err_j^2 / 2, row by row
    for i in range(W.shape[0]):
        _, incr = O.obs_bruteforce_row(W[i], H, bits, group, sym, zero_in_range=zr)
        np.testing.assert_allclose(incr, 0.5 * r["err"][i] ** 2, rtol=1e-9, atol=1e-15)
        np.testing.assert_allclose(incr.sum(), 0.5 * r["err_sq"][i], rtol=1e-10, atol=1e-15)


@pytest.mark.parametrize("group,sym,act", [(0, True, False), (16, True, False), (16, False, False),
                                           (16, True, True)])
def test_total_error_closed_form(group, sym, act):
    """P-3: per row (q - w0) H (q - w0)^T = sum_j err_j^2 with the damped, dead-fixed H."""
    rng = _rng(20 + group)
    d = 48
    X = rng.standard_normal((200, d)) * np.exp(rng.standard_normal(d))
    X[:, 5] = 0.0
    W = rng.standard_normal((7, d)) * 0.05
    H = O.hessian(X)
    U, perm, dead = O.prepare(H, 0.01, act, np.diag(O.xtx(X)))
    r = O.gptq_quantize(W, U, perm, dead, 3, group, sym)
    W0 = W.copy()
    W0[:, dead] = 0
    Hp = H[perm][:, perm]
    Hd = _damped(Hp)
    loss = O.layer_loss(r["Wq"][:, perm], W0[:, perm], Hd)
    np.testing.assert_allclose(loss, r["err_sq"], rtol=1e-10)


@pytest.mark.parametrize("group,sym", [(0, True), (64, True), (64, False)])
def test_diagonal_hessian_reduces_to_rtn_exactly(group, sym):
    """P-4: X = Hadamard columns gives H = 2I, U diagonal, so GPTQ == RTN bit for bit."""
    spec = synth.XSpec(n=512, d=256, kind="hadamard", dtype="f32")
    X = synth.to_numpy_f64(synth.make_x(spec, 0))
    H = O.hessian(X)
    np.testing.assert_array_equal(H, 2 * np.eye(256))
    W = synth.to_numpy_f64(synth.make_weight(128, 256, 0.1, 7))
    U, perm, dead = O.prepare(H, 0.01, False)
    assert np.count_nonzero(U - np.diag(np.diag(U))) == 0
    g = O.gptq_quantize(W, U, perm, dead, 4, group, sym)
    r = O.rtn_quantize(W, 4, group, sym)
    np.testing.assert_array_equal(g["codes"], r["codes"])
    np.testing.assert_array_equal(g["Wq"], r["Wq"])
    np.testing.assert_array_equal(g["packed"], r["packed"])


def test_heavy_damping_reduces_to_rtn():
    """P-5 ([guide] "When it breaks"): heavy damping makes U nearly diagonal -> RTN codes."""
    wl = synth.workload(0)
    X = synth.to_numpy_f64(synth.make_x(wl.layers[0].x, 5))
    W = synth.to_numpy_f64(synth.make_weight(128, 256, 0.1, 6))
    H = O.hessian(X)
    U, perm, dead = O.prepare(H, 1e8, False)
    g = O.gptq_quantize(W, U, perm, dead, 4, 0, True)
    r = O.rtn_quantize(W, 4, 0, True)
    assert np.count_nonzero(g["codes"] != r["codes"]) == 0


@pytest.mark.parametrize("sym", [True, False])
def test_dead_columns_come_out_zero(sym):
    """P-6: W[:, dead] = 0 before the loop, and the grid represents 0 exactly."""
    spec = synth.XSpec(n=1024, d=256, kind="scaled", dtype="bf16", n_outliers=4,
                       outlier_factor=20.0, dead_frac=0.05)
    X = synth.to_numpy_f64(synth.make_x(spec, 11))
    dead_expected = synth.dead_channels(spec, 11).numpy()
    W = synth.to_numpy_f64(synth.make_weight(64, 256, 0.02, 12))
    H = O.hessian(X)
    U, perm, dead = O.prepare(H, 0.01, False)
    np.testing.assert_array_equal(np.nonzero(dead)[0], dead_expected)
    g = O.gptq_quantize(W, U, perm, dead, 4, 128, sym)
    assert np.all(g["Wq"][:, dead] == 0.0)


def test_gptq_output_error_below_rtn():
    """P-7 ([loop]: output error on X well below plain rounding's), per-row scales."""
    wl = synth.workload(0)
    X = synth.to_numpy_f64(synth.make_x(wl.layers[0].x, synth.x_seed(0, wl.layers[0].x)))
    W = synth.to_numpy_f64(synth.make_weight(128, 256, 0.1, synth.weight_seed(0, "w")))
    for bits in (2, 3, 4):
        g = O.gptq_layer(W, X, bits=bits)
        r = O.rtn_quantize(W, bits, 0, True)
        eg = O.rel_output_error(X, W, g["Wq"])
        er = O.rel_output_error(X, W, r["Wq"])
        assert eg < 0.9 * er, (bits, eg, er)


def test_output_error_identity_through_xtx():
    rng = _rng(4)
    X = rng.standard_normal((50, 6))
    W = rng.standard_normal((3, 6))
    Q = W + 0.01 * rng.standard_normal((3, 6))
    assert np.isclose(O.rel_output_error(X, W, Q), O.rel_output_error_from_xtx(O.xtx(X), W, Q), rtol=1e-12)


def test_clipped_codes_stay_on_grid():
    """[guide] "When it breaks": compensation can push weights past the row scale;
    those are clipped to +-qmax, never beyond."""
    rng = _rng(5)
    X = rng.standard_normal((64, 32)) @ rng.standard_normal((32, 32))
    W = rng.standard_normal((16, 32))
    g = O.gptq_layer(W, X, bits=2)
    assert g["codes"].min() >= -1 and g["codes"].max() <= 1


def test_act_order_is_plain_loop_on_permuted_problem():
    """P-10: act_order equals the plain loop on (W[:, perm], H[perm][:, perm]), unpermuted."""
    rng = _rng(6)
    d = 40
    X = rng.standard_normal((160, d)) * np.exp(rng.standard_normal(d))
    W = rng.standard_normal((9, d)) * 0.05
    g = O.gptq_layer(W, X, bits=3, group=8, act_order=True)
    perm = np.argsort(-np.diag(X.T @ X), kind="stable")
    Hp = O.hessian(X[:, perm])
    U2 = O.upper_cholesky_of_inverse(_damped(Hp))
    r = O.gptq_loop(W[:, perm], U2, 3, 8, True)
    np.testing.assert_array_equal(g["perm"], perm)
    np.testing.assert_allclose(g["Wq"][:, perm], r["Q"], rtol=0, atol=1e-12)
    np.testing.assert_array_equal(g["g_idx"][perm], np.arange(d) // 8)


# ------------------------------------------------------------ AutoGPTQ page fixture

def test_auto_page_demo_printed_values():
    """P-8: the AutoGPTQ page's seeded one-row demo prints GPTQ MSE 0.000135, naive
    0.000086, ratio 1.56 — this pins the asymmetric quantizer (half-to-even, zero clamp,
    group-start scale from updated weights)."""
    torch = pytest.importorskip("torch")
    gold = json.load(open(os.path.join(GOLDEN, "auto_demo.json")))
    torch.manual_seed(gold["setup"]["seed"])
    Wt = torch.randn(128, 256) * 0.1
    Xt = torch.randn(512, 256)
    W = Wt.double().numpy()
    X = Xt.double().numpy()
    Hinv = np.linalg.inv(O.auto_compute_hessian(X))
    codes, params = O.auto_gptq_quantize_row(W[0], Hinv, 4, 128)
    deq = O.auto_dequantize_row(codes, params, 128)
    mse = float(np.mean((W[0] - deq) ** 2))
    naive = O.rtn_quantize(W[:1], 4, 0, False, scale_dtype=None)
    naive_mse = float(np.mean((W[0] - naive["Wq"][0]) ** 2))
    p = gold["printed"]
    assert round(mse, 6) == p["gptq_mse"]
    assert round(naive_mse, 6) == p["naive_mse"]
    assert round(mse / naive_mse, 2) == p["ratio"]


# ------------------------------------------------------------ comparison machinery

def test_teacher_forcing_accepts_ties_and_rejects_real_mismatches():
    # codes decided exactly at a half-point: 0.0625 / 0.125 = 0.5 -> 0 (half-to-even)
    W = np.array([[0.875, 0.0625, 0.3]])
    U = np.eye(3)
    r = O.gptq_loop(W, U, 4, 0, True)
    assert r["codes"][0, 1] == 0
    forced = r["codes"].copy()
    forced[0, 1] = 1                       # the other side of the tie: accepted
    r2 = O.gptq_loop(W, U, 4, 0, True, forced_codes=forced)
    assert r2["codes"][0, 1] == 1 and len(r2["ties"]) == 1
    forced = r["codes"].copy()
    forced[0, 2] += 1                      # 0.3/0.125 = 2.4: not a tie -> rejected
    with pytest.raises(O.TieMismatch):
        O.gptq_loop(W, U, 4, 0, True, forced_codes=forced)


def test_perm_equivalent():
    keys = np.array([5.0, 3.0, 3.0000001, 1.0])
    assert O.perm_equivalent([0, 2, 1, 3], [0, 1, 2, 3], keys, 1e-6)
    assert not O.perm_equivalent([0, 3, 1, 2], [0, 1, 2, 3], keys, 1e-6)


# ------------------------------------------------------------ the stored form and its consumer

def test_unpack_by_hand():
    # 4-bit: word 0x76543210 holds codes 0..7 least significant nibble first
    np.testing.assert_array_equal(O.unpack_rows(np.array([[0x76543210]], dtype=np.uint32), 4, 8),
                                  [[0, 1, 2, 3, 4, 5, 6, 7]])
    # 3-bit: codes 5, 6, 7, ... ; code 10 straddles words 0 and 1 (stream bits 30..32)
    u = np.array([[5, 6, 7, 1, 0, 2, 3, 4, 5, 6, 7, 1]])
    stream = [(int(u[0, c]) >> b) & 1 for c in range(12) for b in range(3)]
    words = [sum(bit << p for p, bit in enumerate(stream[32 * w:32 * w + 32])) for w in range(2)]
    np.testing.assert_array_equal(O.unpack_rows(np.array([words], dtype=np.uint32), 3, 12), u)


@pytest.mark.parametrize("bits,d", [(2, 64), (3, 100), (4, 33), (3, 96)])
def test_unpack_inverts_pack(bits, d):
    rng = np.random.default_rng(bits * 1000 + d)
    u = rng.integers(0, 2 ** bits, size=(7, d))
    np.testing.assert_array_equal(O.unpack_rows(O.pack_rows(u, bits), bits, d), u)


@pytest.mark.parametrize("bits,group,sym,act", [(4, 128, True, False), (3, 32, False, True), (2, 0, True, True),
                                                (4, 64, False, False)])
def test_stored_form_dequantises_to_the_loop_weights(bits, group, sym, act):
    """The packed codes, scales, zeros and g_idx the layer returns, read back through
    g_idx, give exactly the dequantised weights of the column loop (in the original
    column order)."""
    rng = np.random.default_rng(bits + group)
    X = rng.standard_normal((400, 256)) * np.exp(rng.standard_normal(256))
    W = 0.05 * rng.standard_normal((24, 256))
    out = O.gptq_layer(W, X, bits, group, sym, 0.01, act)
    G = out["scales"].shape[1]
    zeros = out["zeros"] if not sym else np.full((24, G), 2 ** (bits - 1))
    Wq = O.dequant_stored(out["packed"], out["scales"], zeros, out["g_idx"], bits, 256)
    np.testing.assert_array_equal(Wq, out["Wq"])


def test_dequant_matmul_brute_force():
    rng = np.random.default_rng(5)
    T, d, o, bits, G = 3, 12, 4, 3, 3
    u = rng.integers(0, 8, size=(o, d))
    s = rng.uniform(0.5, 2.0, size=(o, G))
    z = rng.integers(0, 8, size=(o, G))
    g = rng.integers(0, G, size=d)
    X = rng.standard_normal((T, d))
    Y = O.dequant_matmul(X, O.pack_rows(u, bits), s, z, g, bits)
    for t in range(T):
        for r in range(o):
            want = sum(X[t, k] * s[r, g[k]] * (u[r, k] - z[r, g[k]]) for k in range(d))
            assert abs(Y[t, r] - want) <= 1e-12 * (1 + abs(want))


# ------------------------------------------------------------------ layer-wise application

def test_round_bf16_by_hand():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9, -2.5, 0.0, 1.0 + 2 ** -7])
    # 1+2^-8 is a tie between 1 and 1+2^-7 -> even (1); 1+3*2^-8 ties -> even (1+2^-6)
    np.testing.assert_array_equal(O.round_bf16(x), [1.0, 1.0, 1.0 + 2 ** -6, 1.0, -2.5, 0.0, 1.0 + 2 ** -7])


def test_layerwise_first_layer_is_the_plain_layer_and_later_layers_see_quantised_inputs():
    """Layer 0 is calibrated on X itself; layer i on the forward pass through the already
    quantised layers 0..i-1 (not through the original weights)."""
    rng = np.random.default_rng(21)
    X = rng.standard_normal((300, 32))
    Ws = [rng.standard_normal((48, 32)) / np.sqrt(32), rng.standard_normal((40, 48)) / np.sqrt(48),
          rng.standard_normal((8, 40)) / np.sqrt(40)]
    fn = lambda W, h: O.gptq_layer(W, h, 3, 0, True)["Wq"]
    Qs, hs, out = O.apply_layerwise(X, Ws, fn)
    np.testing.assert_array_equal(Qs[0], fn(Ws[0], X))
    h1 = np.maximum(X @ Qs[0].T, 0.0)
    np.testing.assert_array_equal(hs[1], h1)
    np.testing.assert_array_equal(Qs[1], fn(Ws[1], h1))
    assert not np.array_equal(hs[1], np.maximum(X @ Ws[0].T, 0.0))
    np.testing.assert_allclose(out, O.mlp_forward(X, Qs), rtol=1e-12, atol=1e-12)
    # skip_last leaves the output layer in full precision
    Qs2, _, _ = O.apply_layerwise(X, Ws, fn, skip_last=True)
    np.testing.assert_array_equal(Qs2[2], Ws[2])


def test_layerwise_gptq_beats_rtn_end_to_end():
    """The guide page's simulation claim, on a small synthetic MLP with correlated inputs:
    layer-wise GPTQ leaves a smaller output error than layer-wise RTN."""
    rng = np.random.default_rng(22)
    Z = rng.standard_normal((1024, 64))
    X = Z @ rng.standard_normal((64, 64)) / 8.0
    Ws = [rng.standard_normal((128, 64)) / 8.0, rng.standard_normal((128, 128)) / np.sqrt(128),
          rng.standard_normal((16, 128)) / np.sqrt(128)]
    ref = O.mlp_forward(X, Ws)
    err = lambda y: float(np.sum((y - ref) ** 2) / np.sum(ref ** 2))
    _, _, y_g = O.apply_layerwise(X, Ws, lambda W, h: O.gptq_layer(W, h, 3, 0, True)["Wq"])
    _, _, y_r = O.apply_layerwise(X, Ws, lambda W, h: O.rtn_quantize(W, 3, 0, True)["Wq"])
    assert err(y_g) < err(y_r)


# ------------------------------------------------------- pruning with the same update

def _corr_layer(seed, d, o, n_mult=4):
    rng = _rng(seed)
    X = rng.standard_normal((n_mult * d, d)) @ rng.standard_normal((d, d))
    H = _damped(O.hessian(X))
    return rng, X, H, rng.standard_normal((o, d)) * 0.1


@pytest.mark.parametrize("d,block,sparsity", [(8, 4, 0.5), (8, 8, 0.25), (6, 4, 0.5)])
def test_prune_loop_equals_bruteforce_obs(d, block, sparsity):
    """The Cholesky-form loop with pruning equals explicit OBS with Gaussian elimination on
    H^-1 given the same mask (the update the pages say pruning reuses)."""
    rng, X, H, W = _corr_layer(40 + d + block, d, 5)
    U = O.upper_cholesky_of_inverse(H)
    r = O.prune_loop(W, U, sparsity, block)
    for i in range(W.shape[0]):
        w = O.obs_prune_bruteforce_row(W[i], H, r["mask"][i])
        np.testing.assert_allclose(r["W"][i], w, rtol=0, atol=1e-12)


def test_prune_mask_counts_zeros_and_loss_closed_form():
    """Per row and block exactly round(sparsity * width) weights are pruned and come out 0;
    the kept ones after the first pruned one are changed by the compensation; and per row
    (q - w0) H (q - w0)^T equals sum_j err_j^2 (the same closed form as the quantiser's, P-3)."""
    rng, X, H, W = _corr_layer(50, 48, 6)
    U = O.upper_cholesky_of_inverse(H)
    r = O.prune_loop(W, U, 0.5, 16)
    for b0 in range(0, 48, 16):
        np.testing.assert_array_equal(r["mask"][:, b0:b0 + 16].sum(axis=1), 8)
    assert np.all(r["W"][r["mask"]] == 0.0)
    # every kept weight after its row's first pruned one has received compensation
    first = r["mask"].argmax(axis=1)
    after = np.arange(48)[None, :] > first[:, None]
    keep = ~r["mask"] & after
    assert np.all(r["W"][keep] != W[keep])
    D = r["W"] - W
    np.testing.assert_allclose(np.einsum("ij,jk,ik->i", D, H, D), r["err_sq"], rtol=1e-10)


def test_prune_zero_sparsity_is_identity():
    rng, X, H, W = _corr_layer(51, 32, 4)
    r = O.prune_loop(W, O.upper_cholesky_of_inverse(H), 0.0, 16)
    np.testing.assert_array_equal(r["W"], W)
    assert not r["mask"].any()


def test_prune_with_diagonal_hessian_is_magnitude_pruning():
    """X = Hadamard columns gives H = 2I (U diagonal): no compensation reaches other columns,
    so the result is W with each row-block's smallest-|w| half set to 0."""
    spec = synth.XSpec(n=64, d=32, kind="hadamard", dtype="f32")
    X = synth.to_numpy_f64(synth.make_x(spec, 0, device="cpu"))
    H = O.hessian(X)
    np.testing.assert_allclose(H, 2.0 * np.eye(32), atol=0)
    W = _rng(52).standard_normal((5, 32))
    r = O.prune_loop(W, O.upper_cholesky_of_inverse(H), 0.5, 8)
    ref = W.copy()
    for b0 in range(0, 32, 8):
        blk = ref[:, b0:b0 + 8]
        small = np.argsort(np.abs(blk), axis=1, kind="stable")[:, :4]
        np.put_along_axis(blk, small, 0.0, axis=1)
    np.testing.assert_allclose(r["W"], ref, rtol=0, atol=1e-15)


def test_prune_compensation_beats_plain_masking():
    """On correlated inputs the compensated result has a smaller output error than the same
    mask applied without the update (the pages' claim for the update, on pruning)."""
    rng, X, H, W = _corr_layer(53, 64, 16)
    U = O.upper_cholesky_of_inverse(H)
    r = O.prune_loop(W, U, 0.5, 32)
    plain = np.where(r["mask"], 0.0, W)
    assert O.rel_output_error(X, W, r["W"]) < 0.8 * O.rel_output_error(X, W, plain)


def test_prune_layer_permutation_and_dead():
    """prune_layer = prune_loop on (W[:, perm] with dead columns zeroed), unpermuted."""
    rng, X, H, W = _corr_layer(54, 24, 5)
    X[:, 3] = 0.0
    Hd = O.hessian(X)
    U, perm, dead = O.prepare(Hd, 0.01, True, np.diag(O.xtx(X)))
    r = O.prune_layer(W, U, perm, dead, 0.5, 8)
    W0 = W.copy()
    W0[:, dead] = 0.0
    r2 = O.prune_loop(W0[:, perm], U, 0.5, 8)
    inv = np.argsort(perm)
    np.testing.assert_array_equal(r["W"], r2["W"][:, inv])
    assert np.all(r["W"][:, dead] == 0.0)


def test_prune_forced_mask_accepts_only_near_ties():
    """Teacher forcing of the pruning mask: the oracle's own mask forced back changes nothing;
    a mask that swaps two weights of exactly equal saliency is adopted (and logged); a mask
    that swaps a clearly smaller weight for a larger one is rejected."""
    rng, X, H, W = _corr_layer(55, 16, 4)
    U = O.upper_cholesky_of_inverse(H)
    r = O.prune_loop(W, U, 0.5, 8)
    same = O.prune_loop(W, U, 0.5, 8, forced_mask=r["mask"])
    np.testing.assert_array_equal(same["W"], r["W"])
    assert same["ties"] == []
    # an exact tie in block 0 of row 0: give the largest pruned weight and the smallest kept
    # weight of that block the same saliency, then force the other choice
    W2 = W.copy()
    sal = O.prune_saliency(W2, U, 0, 8)[0]
    own = O.prune_loop(W2, U, 0.5, 8)["mask"][0, :8]
    p_max = np.nonzero(own)[0][np.argmax(sal[own])]
    k_min = np.nonzero(~own)[0][np.argmin(sal[~own])]
    W2[0, k_min] = np.sign(W2[0, k_min]) * np.sqrt(sal[p_max]) * U[k_min, k_min]
    base = O.prune_loop(W2, U, 0.5, 8)
    fm = base["mask"].copy()
    a, b = (p_max, k_min) if base["mask"][0, p_max] else (k_min, p_max)
    fm[0, a], fm[0, b] = False, True
    forced = O.prune_loop(W2, U, 0.5, 8, forced_mask=fm)
    assert forced["mask"][0, b] and not forced["mask"][0, a]
    assert [t[:3] for t in forced["ties"]] == [(0, 0, "mask")]
    # a clear swap: keep the smallest-saliency weight, prune the largest
    fm = r["mask"].copy()
    sal = O.prune_saliency(W, U, 0, 8)[1]
    lo_, hi_ = int(np.argmin(sal)), int(np.argmax(sal))
    fm[1, lo_], fm[1, hi_] = False, True
    with pytest.raises(O.TieMismatch):
        O.prune_loop(W, U, 0.5, 8, forced_mask=fm)
