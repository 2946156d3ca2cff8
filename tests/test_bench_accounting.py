"""bench.py's algorithmic work per kernel class (the numerators of its roofline fractions):
the factorisation's chain and side-stream classes add up to the factorisation's total,
every product counted once, and inputs shared by several layers count their Hessian and
factorisation once."""
import types

import pytest

import bench

NB = 128


def _layer(n, d, rows, bits=4, damp=0.01, act_order=False, X=None):
    X = X or types.SimpleNamespace(shape=(n, d))
    spec = types.SimpleNamespace(q=types.SimpleNamespace(bits=bits, damp=damp, act_order=act_order))
    return types.SimpleNamespace(X=X, Wcat=types.SimpleNamespace(shape=(rows, X.shape[1])), spec=spec)


def _prepare_total(d):
    tot = 0.0
    for k0 in range(0, d, NB):
        nb = min(NB, d - k0)
        m = d - k0 - nb
        ncols = k0 + nb
        tot += 2.0 * m * nb * nb + 2.0 * (m * (m + 1) / 2) * nb + 2.0 * nb * ncols * nb + 2.0 * m * ncols * nb
    return tot


@pytest.mark.parametrize("d", [256, 768, 2048, 2100, 4096, 14336])
def test_chain_and_side_add_up_to_the_factorisation(d):
    work = bench.algorithmic([_layer(1024, d, 64)])
    total = _prepare_total(d)
    chain, side = work["tc_gemm_nt_kernel[chain]"], work["tc_gemm_nt_kernel[prepare]"]
    assert chain > 0 and side > 0
    assert chain + side == pytest.approx(total, rel=1e-12)
    # the leading term of the total is 2 d^3 / 3 (the per-panel terms are O(d^2 * 128))
    if d >= 4096:
        assert total == pytest.approx(2.0 * d ** 3 / 3, rel=0.1)


def test_chain_share_by_hand():
    # d = 256 (one-panel super-panels): panel 0 solves m = 128 rows and updates the next
    # panel's 128 columns (lower part) with K = 128; panel 1 has no rows below it
    d = 256
    m, nn, n = 128, 128, 128
    expect = 2.0 * m * n * n + 2.0 * n * (m * nn - nn * (nn - 1) / 2)
    assert bench.algorithmic([_layer(512, d, 8)])["tc_gemm_nt_kernel[chain]"] == pytest.approx(expect)
    # d = 2048 (super-panels of 4): the last panel of a super-panel updates the next panel's
    # columns with all four panels' L21 (K = 512)
    d = 2048
    expect = 0.0
    for k0 in range(0, d, NB):
        m = d - k0 - NB
        if m <= 0:
            continue
        sp0 = k0 // 512 * 512
        ks = 512 if k0 + NB == min(d, sp0 + 512) else NB
        expect += 2.0 * m * NB * NB + 2.0 * ks * (m * NB - NB * (NB - 1) / 2)
    assert bench.algorithmic([_layer(512, d, 8)])["tc_gemm_nt_kernel[chain]"] == pytest.approx(expect)


def test_shared_input_counts_its_hessian_and_factorisation_once():
    X = types.SimpleNamespace(shape=(4096, 1024))
    one = bench.algorithmic([_layer(0, 0, 512, X=X)])
    three = bench.algorithmic([_layer(0, 0, 512, bits=b, X=X) for b in (2, 3, 4)])
    for k in ("hessian_tc_kernel", "tc_gemm_nt_kernel[chain]", "tc_gemm_nt_kernel[prepare]", "potrf_diag_kernel"):
        assert three[k] == pytest.approx(one[k])
    for k in ("gptq_block_kernel", "tc_gemm_nt_kernel[trailing]", "init_work_kernel"):
        assert three[k] == pytest.approx(3 * one[k])


class _Ev:
    """A stand-in for a CUDA event: a time stamp in ms."""

    def __init__(self, t):
        self.t = t

    def elapsed_time(self, other):
        return other.t - self.t


def test_stage_breakdown_per_group_and_bits():
    # two groups: input A read by layers 0 (2 bits) and 1 (4 bits); input B by layer 2 (4
    # bits). One step: A's H 10 ms, U 4 ms, quantisations 3 and 5 ms; B's H 20, U 6, q 7.
    XA = types.SimpleNamespace(shape=(100, 64))
    XB = types.SimpleNamespace(shape=(100, 32))

    def lay(X, bits, name):
        return types.SimpleNamespace(X=X, names=[name], spec=types.SimpleNamespace(q=types.SimpleNamespace(bits=bits)))

    layers = [lay(XA, 2, "a2"), lay(XA, 4, "a4"), lay(XB, 4, "b4")]
    groups = [[0, 1], [2]]
    ev = lambda *ts: [_Ev(t) for t in ts]
    a = ev(0, 10, 14, 22) + [(0, _Ev(17)), (1, _Ev(22))]
    b = ev(22, 42, 48, 55) + [(2, _Ev(55))]
    per_group, per_bits = bench.stage_breakdown([a, b], groups, layers, steps=1)
    assert per_group[0]["hessian"] == 10 and per_group[0]["prepare"] == 4
    assert per_group[0]["quantize"] == {"2b a2": 3, "4b a4": 5}
    assert per_group[1]["quantize"] == {"4b b4": 7}
    assert per_bits["2"] == {"quantize": 3, "fresh": 3 + 14, "amortised": 3 + 14 / 2}
    assert per_bits["4"] == {"quantize": 12, "fresh": 12 + 14 + 26, "amortised": 12 + 14 / 2 + 26}
