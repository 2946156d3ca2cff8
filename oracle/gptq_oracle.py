"""Plain CPU fp64 restatement of GPTQ's per-layer quantization (test infrastructure only).

This module is the oracle the CUDA path is checked against. It is written for a
reader who checks it against the pages by eye: no blocking, no fusion, no
reordering beyond what the pages state. All floating point is NumPy float64
unless a function says otherwise.

Sources, cited by page title and section:

* [loop]  "GPTQ's error-compensation loop" (exercise page): the four-step column
          algorithm, `hessian_inverse_chol`, `quantize_column`, and the solution.
* [auto]  "GPTQ > Implementation with AutoGPTQ": `compute_hessian`, the
          `quantize_weight`/`dequantize_weight` primitives, `gptq_quantize_row` and
          its seeded one-row demo.
* [guide] "GPTQ" (guide page): "How it works" (OBS step, Gaussian elimination,
          the two tricks, damping), "The code, line by line", "When it breaks" and
          "Source code" (`gptq`, `_hessian_inverse_chol`).

Readings taken where the pages are silent or disagree (each also listed in the
design notes):

* Hessian scale and damping follow [loop]/[guide] (2 X^T X / n, relative damping
  0.01 * mean(diag H)), not [auto]'s absolute 1e-4 (kept only for its fixture).
* qmax for the symmetric grid is 2^(bits-1) - 1 ([loop] solution), so 2 bits is the
  ternary grid {-s, 0, s} ([guide] "What the simulations show").
* The asymmetric quantizer is [auto]'s min/max + zero point, evaluated per (row,
  group) at the group start from the updated weights, as [guide] does for its
  symmetric group scales.
* Scales are stored as float32; the grid a weight is rounded onto is the stored
  scale (so dequantised = code * stored scale exactly). `scale_dtype=None` keeps
  the pages' unrounded float64 scale.
* act_order: the permutation is a *stable* descending sort of diag(X^T X) (ties
  by ascending channel index); the permuted Hessian is H[perm][:, perm], which
  equals the Hessian of X[:, perm] that [guide]'s code recomputes.
* Symmetric codes are stored as unsigned u = code + 2^(bits-1) with zero point
  2^(bits-1); packing is an LSB-first bitstream of `bits`-bit u per row in 32-bit
  words (the pages give no layout).
"""
from __future__ import annotations

import math
from typing import Dict, Iterable, Optional, Sequence, Tuple

import numpy as np

F64 = np.float64

__all__ = [
    "xtx", "hessian_accumulate", "hessian_from_sum", "hessian",
    "dead_mask", "fix_dead", "add_damping", "upper_cholesky_of_inverse", "act_order_perm",
    "prepare", "qmax_sym", "maxq_asym", "sym_params", "asym_params", "quant_codes", "dequant",
    "gptq_loop", "gptq_quantize", "gptq_layer", "rtn_quantize", "unsigned_codes", "pack_rows",
    "g_idx_for", "rel_output_error", "rel_output_error_from_xtx", "layer_loss",
    "obs_bruteforce_row", "auto_compute_hessian", "auto_gptq_quantize_row", "auto_dequantize_row",
    "near_half", "perm_equivalent", "TieMismatch", "unpack_rows", "dequant_stored", "dequant_matmul",
    "round_bf16", "mlp_forward", "apply_layerwise",
    "prune_saliency", "prune_loop", "prune_layer", "obs_prune_bruteforce_row",
]


# ----------------------------------------------------------------------------------------
# Hessian  ([loop] statement and `hessian_inverse_chol`; [guide] "Source code",
#           `_hessian_inverse_chol`, first line: H = 2 X^T X / n)
# ----------------------------------------------------------------------------------------

def xtx(X) -> np.ndarray:
    """S = X^T X in float64 (the unscaled Gram matrix of the calibration rows)."""
    X = np.asarray(X, dtype=F64)
    return X.T @ X


def hessian_accumulate(batches: Iterable) -> Tuple[np.ndarray, int]:
    """Stream S = sum_b X_b^T X_b over token batches; returns (S, n)."""
    S = None
    n = 0
    for Xb in batches:
        Xb = np.asarray(Xb, dtype=F64)
        S = xtx(Xb) if S is None else S + xtx(Xb)
        n += Xb.shape[0]
    return S, n


def hessian_from_sum(S, n: int) -> np.ndarray:
    """H = 2 S / n: the curvature of the layer's squared output error."""
    return 2.0 * np.asarray(S, dtype=F64) / n


def hessian(X) -> np.ndarray:
    """H = 2 X^T X / n for the (n, d) calibration rows X."""
    X = np.asarray(X, dtype=F64)
    return hessian_from_sum(xtx(X), X.shape[0])


# ----------------------------------------------------------------------------------------
# Preparation: dead inputs, damping, U  ([guide] "Source code", `_hessian_inverse_chol`;
#   "The code, line by line"; "How it works", Damping; [loop] `hessian_inverse_chol`)
# ----------------------------------------------------------------------------------------

def dead_mask(H) -> np.ndarray:
    """Inputs that never activate: diag(H) == 0."""
    return np.diag(np.asarray(H)) == 0


def fix_dead(H) -> np.ndarray:
    """Copy of H with H[j, j] = 1 for every dead j (keeps H invertible)."""
    H = np.array(H, dtype=F64, copy=True)
    dead = dead_mask(H)
    H[dead, dead] = 1.0          # paired boolean indexing: diagonal entries only
    return H


def add_damping(H, damp: float) -> np.ndarray:
    """H + damp * mean(diag H) * I (the mean is taken as H stands, i.e. after the dead fix)."""
    H = np.asarray(H, dtype=F64)
    return H + damp * np.mean(np.diag(H)) * np.eye(H.shape[0])


def upper_cholesky_of_inverse(H) -> np.ndarray:
    """U, the upper Cholesky factor of H^-1 (H^-1 = U^T U): numpy's lower factor, transposed."""
    return np.linalg.cholesky(np.linalg.inv(np.asarray(H, dtype=F64))).T


def act_order_perm(diag_xtx) -> np.ndarray:
    """Columns with the largest activations first: stable argsort of -diag(X^T X)."""
    return np.argsort(-np.asarray(diag_xtx, dtype=F64), kind="stable")


def prepare(H, damp: float = 0.01, act_order: bool = False,
            diag_xtx=None) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """(U, perm, dead) for one layer, in the order [guide]'s `gptq` takes the steps.

    dead comes from the unpermuted H. With act_order, perm sorts diag(X^T X)
    (`diag_xtx`, default diag(H), same order) and U is formed from the permuted H.
    U is in the loop's (permuted) column order; perm is the identity without act_order.
    """
    H = np.asarray(H, dtype=F64)
    d = H.shape[0]
    dead = dead_mask(H)
    perm = np.arange(d)
    if act_order:
        perm = act_order_perm(np.diag(H) if diag_xtx is None else diag_xtx)
        H = H[perm][:, perm]
    Hd = add_damping(fix_dead(H), damp)
    U = upper_cholesky_of_inverse(Hd)
    return U, perm, dead


# ----------------------------------------------------------------------------------------
# Quantizers
#   symmetric:  [loop] `quantize_column`, [guide] "Source code" (per-row scale from the
#               starting W; group scales from the updated W at each group start)
#   asymmetric: [auto] `quantize_weight`, `dequantize_weight` and the group-start
#               parameter block of `gptq_quantize_row`
# ----------------------------------------------------------------------------------------

def qmax_sym(bits: int) -> int:
    return 2 ** (bits - 1) - 1


def maxq_asym(bits: int) -> int:
    return 2 ** bits - 1


def _stored(x, scale_dtype):
    x = np.asarray(x, dtype=F64)
    return x if scale_dtype is None else x.astype(scale_dtype).astype(F64)


def sym_params(block, qmax: int, scale_dtype=np.float32):
    """Per-row scale max(max_j |w_j|, 1e-12) / qmax over the columns of `block`; zero point 0."""
    block = np.asarray(block, dtype=F64)
    scale = _stored(np.maximum(np.abs(block).max(axis=1), 1e-12) / qmax, scale_dtype)
    return scale, np.zeros(block.shape[0], dtype=np.int64)


def asym_params(block, maxq: int, scale_dtype=np.float32, zero_in_range: bool = False):
    """Per-row min/max scale and zero point: scale = (max - min) / maxq (1.0 if max == min),
    zero = clamp(round(-min / scale), 0, maxq).

    zero_in_range: the variant whose range is first widened to contain 0,
    min <- min(min, 0), max <- max(max, 0), so that 0 is a grid point (z lands in
    [0, maxq] unclamped and dequantises to exactly 0). Not on the pages, which take the
    raw min/max; this is the plain reading of "the range includes 0"."""
    block = np.asarray(block, dtype=F64)
    mn = block.min(axis=1)
    mx = block.max(axis=1)
    if zero_in_range:
        mn = np.minimum(mn, 0.0)
        mx = np.maximum(mx, 0.0)
    scale = np.where(mx > mn, (mx - mn) / maxq, 1.0)
    scale = _stored(scale, scale_dtype)
    zero = np.clip(np.round(-mn / scale), 0, maxq).astype(np.int64)
    return scale, zero


def _pre_round(w, scale, zero, sym: bool):
    return w / scale if sym else w / scale + zero


def quant_codes(w, scale, zero, bits: int, sym: bool) -> np.ndarray:
    """Integer codes: sym clip(round(w/s), -qmax, qmax); asym clip(round(w/s + z), 0, maxq).
    Rounding is half-to-even (np.round)."""
    t = _pre_round(np.asarray(w, F64), scale, zero, sym)
    if sym:
        q = qmax_sym(bits)
        return np.clip(np.round(t), -q, q).astype(np.int64)
    return np.clip(np.round(t), 0, maxq_asym(bits)).astype(np.int64)


def dequant(codes, scale, zero, sym: bool) -> np.ndarray:
    """sym: code * s;  asym: s * (code - z)."""
    codes = np.asarray(codes, dtype=F64)
    return codes * scale if sym else scale * (codes - zero)


def near_half(t, tol: float) -> np.ndarray:
    """True where t lies within `tol` of a half-integer (a rounding decision point)."""
    t = np.asarray(t, dtype=F64)
    return np.abs(t - np.floor(t) - 0.5) <= tol


class TieMismatch(AssertionError):
    """A forced code differs from the oracle's outside the allowed half-point band."""


def _force(own, forced, t, lo, hi, tol, what, j, log):
    """Adopt `forced` where it differs from `own`, if the oracle's pre-rounding value t is
    within `tol` of the half-point between the two codes; otherwise raise."""
    bad = np.nonzero(forced != own)[0]
    if bad.size == 0:
        return own
    tb = t[bad]
    lower = np.clip(np.floor(tb), lo, hi)
    upper = np.clip(np.floor(tb) + 1, lo, hi)
    ok = near_half(tb, tol) & ((forced[bad] == lower) | (forced[bad] == upper))
    if not np.all(ok):
        i = bad[np.argmin(ok)]
        raise TieMismatch(f"{what} mismatch at row {i}, column {j}: oracle {own[i]} (pre-round "
                          f"{t[i]!r}), forced {forced[i]}")
    for i in bad:
        log.append((int(i), int(j), what, float(t[i])))
    out = own.copy()
    out[bad] = forced[bad]
    return out


def gptq_loop(W, U, bits: int, group: int = 0, sym: bool = True, scale_dtype=np.float32,
              forced_codes=None, forced_zeros=None, tie_tol: float = 1e-4,
              zero_in_range: bool = False) -> Dict[str, np.ndarray]:
    """GPTQ's fixed-order column loop on an already dead-zeroed, already permuted W.

    For j = 0 .. d-1 ([loop] algorithm; [guide] "Source code", `gptq` loop):
      at a group start (group > 0, j % group == 0) the scale (and zero point) come from
      the updated W[:, j:j+group]; without groups they come once from the starting W;
      q = quantised column j;  err = (W[:, j] - q) / U[j, j];
      W[:, j+1:] -= outer(err, U[j, j+1:]).
    Returns integer codes, dequantised Q, per-group scales/zeros, and per-row sum err^2.

    Teacher forcing: if `forced_codes` (and for asym `forced_zeros`) are given, each
    decision that differs from the oracle's own is accepted only where the oracle's
    pre-rounding value is within `tie_tol` of the half-point between the two codes;
    the forced value is then adopted and the loop continues. Accepted mismatches are
    returned in 'ties'.
    """
    W = np.array(W, dtype=F64, copy=True)
    U = np.asarray(U, dtype=F64)
    o, d = W.shape
    G = -(-d // group) if group else 1
    qm = qmax_sym(bits) if sym else maxq_asym(bits)
    lo, hi = (-qm, qm) if sym else (0, qm)
    params = ((lambda b: sym_params(b, qm, scale_dtype)) if sym
              else (lambda b: asym_params(b, qm, scale_dtype, zero_in_range)))

    codes = np.zeros((o, d), dtype=np.int64)
    Q = np.zeros((o, d), dtype=F64)
    scales = np.zeros((o, G), dtype=F64)
    zeros = np.zeros((o, G), dtype=np.int64)
    err_sq = np.zeros(o, dtype=F64)
    errs = np.zeros((o, d), dtype=F64)
    ties = []

    def take_params(block, gi, j):
        scale, zero = params(block)
        if not sym and forced_zeros is not None:
            mn = np.asarray(block, F64).min(axis=1)
            zero = _force(zero, np.asarray(forced_zeros)[:, gi].astype(np.int64), -mn / scale,
                          0, qm, tie_tol, "zero", j, ties)
        scales[:, gi] = scale
        zeros[:, gi] = zero
        return scale, zero

    scale = zero = None
    if not group:
        scale, zero = take_params(W, 0, 0)      # per row, from the starting weights
    for j in range(d):
        if group and j % group == 0:            # group scales use the *updated* weights
            scale, zero = take_params(W[:, j:j + group], j // group, j)
        w = W[:, j]
        c = quant_codes(w, scale, zero, bits, sym)
        if forced_codes is not None:
            c = _force(c, np.asarray(forced_codes)[:, j].astype(np.int64),
                       _pre_round(w, scale, zero, sym), lo, hi, tie_tol, "code", j, ties)
        q = dequant(c, scale, zero, sym)
        codes[:, j] = c
        Q[:, j] = q
        err = (w - q) / U[j, j]
        W[:, j + 1:] -= np.outer(err, U[j, j + 1:])
        err_sq += err ** 2
        errs[:, j] = err
    return {"codes": codes, "Q": Q, "scales": scales, "zeros": zeros, "err_sq": err_sq, "err": errs,
            "ties": ties}


def unsigned_codes(codes, bits: int, sym: bool) -> np.ndarray:
    """Codes as stored unsigned values: sym u = code + 2^(bits-1); asym u = code."""
    codes = np.asarray(codes, dtype=np.int64)
    return codes + (2 ** (bits - 1) if sym else 0)


def g_idx_for(perm, group: int, d: int) -> np.ndarray:
    """Column -> group index ([guide] "When it breaks": act_order with groups needs g_idx):
    the column quantised at loop position k belongs to group k // group."""
    g = np.zeros(d, dtype=np.int64)
    if group:
        perm = np.arange(d) if perm is None else np.asarray(perm)
        g[perm] = np.arange(d) // group
    return g


def pack_rows(ucodes, bits: int) -> np.ndarray:
    """Per row, an LSB-first bitstream of `bits`-bit unsigned codes in 32-bit words.

    Code c of a row occupies stream bits [c*bits, (c+1)*bits), least significant bit
    first; stream bit p is bit (p % 32) of word p // 32. Rows are padded with zero bits
    to a whole number of words.
    """
    u = np.asarray(ucodes, dtype=np.int64)
    o, d = u.shape
    nbits = d * bits
    nwords = -(-nbits // 32)
    stream = np.zeros((o, nwords * 32), dtype=np.int64)
    for b in range(bits):
        stream[:, b:nbits:bits] = (u >> b) & 1
    weights = np.array([1 << k for k in range(32)], dtype=np.int64)
    words = (stream.reshape(o, nwords, 32) * weights).sum(axis=2)
    return words.astype(np.uint32)


def unpack_rows(packed, bits: int, d: int) -> np.ndarray:
    """The d unsigned `bits`-bit codes of each row of a pack_rows bitstream: code c is
    stream bits [c*bits, (c+1)*bits), stream bit p being bit (p % 32) of word p // 32."""
    w = np.asarray(packed).astype(np.uint32).astype(np.int64)
    o = w.shape[0]
    stream = (w[:, :, None] >> np.arange(32, dtype=np.int64)) & 1
    stream = stream.reshape(o, -1)[:, : d * bits]
    u = np.zeros((o, d), dtype=np.int64)
    for b in range(bits):
        u |= stream[:, b::bits] << b
    return u


def dequant_stored(packed, scales, zeros, g_idx, bits: int, d: int) -> np.ndarray:
    """The weights a consumer of the stored form sees: Wq[o][k] = s[o][g] * (u[o][k] -
    z[o][g]) with g = g_idx[k] ([auto] `dequantize_weight`: scale * (code - zero); [guide]
    "When it breaks": with act_order a kernel needs the stored column-to-group index).
    Symmetric codes are stored as u = code + 2^(bits-1) with zero 2^(bits-1), so this is
    scale * code for them."""
    u = unpack_rows(packed, bits, d).astype(F64)
    g = np.asarray(g_idx, dtype=np.int64)
    s = np.asarray(scales, dtype=F64)[:, g]
    z = np.asarray(zeros, dtype=F64)[:, g]
    return s * (u - z)


def dequant_matmul(X, packed, scales, zeros, g_idx, bits: int) -> np.ndarray:
    """Y = X Wq^T in fp64 with Wq from the stored form (dequant_stored)."""
    X = np.asarray(X, dtype=F64)
    return X @ dequant_stored(packed, scales, zeros, g_idx, bits, X.shape[1]).T


def gptq_quantize(W, U, perm, dead, bits: int, group: int = 0, sym: bool = True,
                  scale_dtype=np.float32, forced_codes=None, forced_zeros=None,
                  tie_tol: float = 1e-4, zero_in_range: bool = False) -> Dict[str, np.ndarray]:
    """One layer's quantisation given (U, perm, dead), outputs in the original column order.

    Follows [guide]'s `gptq` after its `_hessian_inverse_chol` call: W[:, dead] = 0,
    columns permuted by perm, the column loop, then Q[:, argsort(perm)].
    `forced_codes` is in the original column order (as the CUDA path returns it).
    """
    W = np.array(W, dtype=F64, copy=True)
    o, d = W.shape
    W[:, np.asarray(dead, dtype=bool)] = 0.0
    perm = np.arange(d) if perm is None else np.asarray(perm)
    fc = None if forced_codes is None else np.asarray(forced_codes)[:, perm]
    r = gptq_loop(W[:, perm], U, bits, group, sym, scale_dtype, fc, forced_zeros, tie_tol, zero_in_range)
    inv = np.argsort(perm)
    u = unsigned_codes(r["codes"][:, inv], bits, sym)
    return {
        "codes": r["codes"][:, inv], "Wq": r["Q"][:, inv], "scales": r["scales"],
        "zeros": (r["zeros"] if not sym else np.full_like(r["zeros"], 2 ** (bits - 1))),
        "g_idx": g_idx_for(perm, group, d), "packed": pack_rows(u, bits),
        "err_sq": r["err_sq"], "ties": r["ties"], "perm": perm,
    }


def gptq_layer(W, X, bits: int = 4, group: int = 0, sym: bool = True, damp: float = 0.01,
               act_order: bool = False, scale_dtype=np.float32) -> Dict[str, np.ndarray]:
    """The whole layer pass of [guide]'s `gptq(Wt, X, bits, group, damp, act_order)`."""
    X = np.asarray(X, dtype=F64)
    S = xtx(X)
    H = hessian_from_sum(S, X.shape[0])
    U, perm, dead = prepare(H, damp, act_order, np.diag(S))
    out = gptq_quantize(W, U, perm, dead, bits, group, sym, scale_dtype)
    out.update({"U": U, "dead": dead, "H": H})
    return out


def round_bf16(a) -> np.ndarray:
    """Round to the nearest bfloat16 (ties to even), returned as fp64: the activations a
    bf16 forward pass hands to the next layer."""
    x = np.asarray(a, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(F64)


def mlp_forward(X, Ws, act_round=None):
    """The MLP of the guide page's simulations: hidden layers relu(h W^T), the last layer
    linear (no biases: the pages give none). `act_round` rounds every layer output."""
    h = np.asarray(X, dtype=F64)
    for i, W in enumerate(Ws):
        h = h @ np.asarray(W, dtype=F64).T
        if i < len(Ws) - 1:
            h = np.maximum(h, 0.0)
        if act_round is not None:
            h = act_round(h)
    return h


def apply_layerwise(X, Ws, fn, skip_last: bool = False, act_round=None):
    """[guide] `apply_layerwise`: run fn(W, layer_input) -> quantised W on every layer in
    order, each calibrated on the inputs it will actually see — the outputs of the layers
    before it, already quantised. Returns the quantised weights, the calibration input of
    every layer and the final output."""
    h = np.asarray(X, dtype=F64)
    if act_round is not None:
        h = act_round(h)
    Qs, hs = [], []
    for i, W in enumerate(Ws):
        hs.append(h)
        Q = np.asarray(W, dtype=F64) if (skip_last and i == len(Ws) - 1) else fn(W, h)
        Qs.append(Q)
        h = h @ Q.T
        if i < len(Ws) - 1:
            h = np.maximum(h, 0.0)
        if act_round is not None:
            h = act_round(h)
    return Qs, hs, h


def rtn_quantize(W, bits: int, group: int = 0, sym: bool = True, dead=None,
                 scale_dtype=np.float32, zero_in_range: bool = False) -> Dict[str, np.ndarray]:
    """Round-to-nearest baseline: every weight rounded on its own onto the same grid
    ([loop] intro; [guide] "The idea"): scales from W itself (per row, or per contiguous
    group), no error feedback. Dead columns are zeroed first when `dead` is given."""
    W = np.array(W, dtype=F64, copy=True)
    o, d = W.shape
    if dead is not None:
        W[:, np.asarray(dead, dtype=bool)] = 0.0
    qm = qmax_sym(bits) if sym else maxq_asym(bits)
    G = -(-d // group) if group else 1
    step = group if group else d
    codes = np.zeros((o, d), dtype=np.int64)
    Wq = np.zeros((o, d), dtype=F64)
    scales = np.zeros((o, G))
    zeros = np.zeros((o, G), dtype=np.int64)
    for gi in range(G):
        sl = slice(gi * step, min(d, (gi + 1) * step))
        s, z = (sym_params(W[:, sl], qm, scale_dtype) if sym
                else asym_params(W[:, sl], qm, scale_dtype, zero_in_range))
        c = quant_codes(W[:, sl], s[:, None], z[:, None], bits, sym)
        codes[:, sl] = c
        Wq[:, sl] = dequant(c, s[:, None], z[:, None], sym)
        scales[:, gi] = s
        zeros[:, gi] = z if not sym else 2 ** (bits - 1)
    u = unsigned_codes(codes, bits, sym)
    return {"codes": codes, "Wq": Wq, "scales": scales, "zeros": zeros,
            "g_idx": g_idx_for(None, group, d), "packed": pack_rows(u, bits)}


# ----------------------------------------------------------------------------------------
# Measurements  ([guide] "What the simulations show": ||h W - h Wq||^2 / ||h W||^2)
# ----------------------------------------------------------------------------------------

def rel_output_error(X, W, Q) -> float:
    """||X W^T - X Q^T||^2 / ||X W^T||^2 for (out, in) weights and (n, in) inputs."""
    X = np.asarray(X, F64)
    Y = X @ np.asarray(W, F64).T
    Yq = X @ np.asarray(Q, F64).T
    return float(np.sum((Y - Yq) ** 2) / np.sum(Y ** 2))


def rel_output_error_from_xtx(S, W, Q) -> float:
    """The same ratio through S = X^T X: tr(D S D^T) / tr(W S W^T), D = W - Q."""
    S = np.asarray(S, F64)
    W = np.asarray(W, F64)
    D = W - np.asarray(Q, F64)
    return float(np.sum((D @ S) * D) / np.sum((W @ S) * W))


def layer_loss(Q, W0, H) -> np.ndarray:
    """Per row (q - w0) H (q - w0)^T ([guide] "How it works": E(w') up to a constant)."""
    D = np.asarray(Q, F64) - np.asarray(W0, F64)
    return np.sum((D @ np.asarray(H, F64)) * D, axis=1)


# ----------------------------------------------------------------------------------------
# Pruning with the same update ([guide] "Going further": SparseGPT reuses the exact same
# update for pruning). The pages give the update only; the mask rule is a reading:
# at the start of each block of columns, in each row, the weights whose removal costs
# least on their own are pruned -- by [guide] "How it works", removing w_j alone raises the
# loss by e^2 / (2 Hinv_F[j, j]) with e = w_j, and in the Cholesky form Hinv_F[j, j] is
# U[j, j]^2, so the saliency is (w_j / U[j, j])^2 (the factor 1/2 dropped). The block's
# weights are the updated ones at the block start, like the group scales of the loop.
# ----------------------------------------------------------------------------------------

def prune_saliency(W, U, j0: int, j1: int) -> np.ndarray:
    """(w_j / U[j, j])^2 for the columns [j0, j1) of W (rows x columns)."""
    W = np.asarray(W, dtype=F64)
    u = np.diag(np.asarray(U, dtype=F64))[j0:j1]
    return (W[:, j0:j1] / u) ** 2


def _force_mask(own, forced, sal, k, tol, b0, log):
    """Adopt the forced mask of one block where it differs from the oracle's own, if in every
    such row it prunes exactly k weights and every weight it prunes that the oracle keeps has
    a saliency within a relative `tol` of the smallest saliency among the weights the oracle
    prunes instead (a near-tie of the ranking); otherwise raise."""
    forced = np.asarray(forced, dtype=bool)
    rows = np.nonzero(np.any(forced != own, axis=1))[0]
    for i in rows:
        extra = forced[i] & ~own[i]       # pruned by the forced mask only
        instead = own[i] & ~forced[i]     # pruned by the oracle only
        if forced[i].sum() != k or sal[i, extra].max() > (1.0 + tol) * sal[i, instead].min():
            raise TieMismatch(f"mask mismatch at row {i}, block at column {b0}: forced prunes "
                              f"{np.nonzero(extra)[0] + b0} (saliency {sal[i, extra]}), oracle "
                              f"{np.nonzero(instead)[0] + b0} (saliency {sal[i, instead]})")
        log.append((int(i), int(b0), "mask", float(sal[i, extra].max() / sal[i, instead].min() - 1.0)))
    out = own.copy()
    out[rows] = forced[rows]
    return out


def prune_loop(W, U, sparsity: float, block: int = 128, forced_mask=None,
               tie_tol: float = 1e-4) -> Dict[str, np.ndarray]:
    """The column loop of [loop] with pruning in place of rounding, on an already dead-zeroed,
    already permuted W: per block of `block` columns, each row prunes its
    round(sparsity * width) lowest-saliency weights (stable order on ties); then for every
    column j: q = 0 where pruned, else w_j; err = (w_j - q) / U[j, j];
    W[:, j+1:] -= outer(err, U[j, j+1:]). Returns the pruned-and-compensated W, the mask and
    per-row sum err^2.

    Teacher forcing (as gptq_loop's for codes): with `forced_mask`, a block whose forced
    mask differs from the oracle's own is accepted only where the difference is a near-tie
    of the saliency ranking (`_force_mask`); the forced mask is then adopted and the loop
    continues. Accepted differences are returned in 'ties'."""
    W = np.array(W, dtype=F64, copy=True)
    U = np.asarray(U, dtype=F64)
    o, d = W.shape
    mask = np.zeros((o, d), dtype=bool)
    err_sq = np.zeros(o, dtype=F64)
    ties = []
    for b0 in range(0, d, block):
        b1 = min(d, b0 + block)
        k = int(round(sparsity * (b1 - b0)))
        if k > 0:
            sal = prune_saliency(W, U, b0, b1)
            idx = np.argsort(sal, axis=1, kind="stable")[:, :k]
            np.put_along_axis(mask[:, b0:b1], idx, True, axis=1)
            if forced_mask is not None:
                mask[:, b0:b1] = _force_mask(mask[:, b0:b1], np.asarray(forced_mask)[:, b0:b1], sal, k, tie_tol,
                                             b0, ties)
        elif forced_mask is not None and np.any(np.asarray(forced_mask)[:, b0:b1]):
            raise TieMismatch(f"mask mismatch: block at column {b0} prunes nothing")
        for j in range(b0, b1):
            q = np.where(mask[:, j], 0.0, W[:, j])
            err = (W[:, j] - q) / U[j, j]
            W[:, j] = q
            W[:, j + 1:] -= np.outer(err, U[j, j + 1:])
            err_sq += err * err
    return {"W": W, "mask": mask, "err_sq": err_sq, "ties": ties}


def prune_layer(W, U, perm, dead, sparsity: float, block: int = 128, forced_mask=None,
                tie_tol: float = 1e-4) -> Dict[str, np.ndarray]:
    """Pruning of one layer given (U, perm, dead) as `gptq_quantize` takes them: W[:, dead] = 0,
    columns permuted, `prune_loop`, results back in the original column order
    (`forced_mask`, if given, is in the original column order)."""
    W = np.array(W, dtype=F64, copy=True)
    o, d = W.shape
    W[:, np.asarray(dead, dtype=bool)] = 0.0
    perm = np.arange(d) if perm is None else np.asarray(perm)
    fm = None if forced_mask is None else np.asarray(forced_mask, dtype=bool)[:, perm]
    r = prune_loop(W[:, perm], U, sparsity, block, fm, tie_tol)
    inv = np.argsort(perm)
    return {"W": r["W"][:, inv], "mask": r["mask"][:, inv], "err_sq": r["err_sq"], "ties": r["ties"]}


def obs_prune_bruteforce_row(w, H, mask):
    """One row pruned by explicit OBS with a given mask: for j in order, the target is 0 where
    masked and w_j (unchanged) elsewhere; e = w_j - target; delta = -(e / Hinv[j, j]) *
    Hinv[j, F] over the remaining coordinates F; then Hinv is eliminated as in
    `obs_bruteforce_row`. Returns the final row."""
    w = np.array(w, dtype=F64, copy=True)
    d = w.shape[0]
    Hinv = np.linalg.inv(np.asarray(H, F64))
    F = list(range(d))
    for j in range(d):
        target = 0.0 if mask[j] else w[j]
        e = w[j] - target
        hjj = Hinv[j, j]
        w[F] = w[F] - (e / hjj) * Hinv[j, F]
        w[j] = target
        Fn = F[1:]
        if Fn:
            sub = Hinv[np.ix_(Fn, Fn)] - np.outer(Hinv[Fn, j], Hinv[j, Fn]) / hjj
            Hinv = np.zeros_like(Hinv)
            Hinv[np.ix_(Fn, Fn)] = sub
        F = Fn
    return w


# ----------------------------------------------------------------------------------------
# Brute-force OBS  ([guide] "How it works": OBS step 1-4, then "Remove j and repeat")
# ----------------------------------------------------------------------------------------

def obs_bruteforce_row(w, H, bits: int, group: int = 0, sym: bool = True, scale_dtype=np.float32,
                       zero_in_range: bool = False):
    """One row through explicit OBS: no Cholesky factor, only H^-1 and elimination.

    For j in order: e = w_j - quant(w_j); delta = -(e / Hinv[j, j]) * Hinv[j, F] over the
    remaining coordinates F (so w_j lands on quant(w_j)); the loss grows by
    e^2 / (2 Hinv[j, j]); then Hinv <- Hinv - Hinv[:, j] Hinv[j, :] / Hinv[j, j],
    restricted to F minus j. Returns (q, per-step loss increments).
    """
    w = np.array(w, dtype=F64, copy=True)
    d = w.shape[0]
    Hinv = np.linalg.inv(np.asarray(H, F64))
    F = list(range(d))
    qm = qmax_sym(bits) if sym else maxq_asym(bits)
    params = ((lambda b: sym_params(b, qm, scale_dtype)) if sym
              else (lambda b: asym_params(b, qm, scale_dtype, zero_in_range)))
    scale, zero = params(w[None, :])
    q = np.zeros(d)
    incr = np.zeros(d)
    for j in range(d):
        if group and j % group == 0:
            scale, zero = params(w[None, j:j + group])
        c = quant_codes(w[j:j + 1], scale, zero, bits, sym)
        qj = dequant(c, scale, zero, sym)[0]
        e = w[j] - qj
        hjj = Hinv[j, j]
        delta = -(e / hjj) * Hinv[j, F]
        w[F] = w[F] + delta
        w[j] = qj
        q[j] = qj
        incr[j] = e * e / (2.0 * hjj)
        Fn = F[1:]
        if Fn:
            sub = Hinv[np.ix_(Fn, Fn)] - np.outer(Hinv[Fn, j], Hinv[j, Fn]) / hjj
            Hinv = np.zeros_like(Hinv)
            Hinv[np.ix_(Fn, Fn)] = sub
        F = Fn
    return q, incr


# ----------------------------------------------------------------------------------------
# [auto]'s variant, kept only as a fixture for the asymmetric quantizer: absolute damping
# 1e-4 on 2 X^T X, and a static (never eliminated) inverse-Hessian column for the update.
# ----------------------------------------------------------------------------------------

def auto_compute_hessian(X) -> np.ndarray:
    """[auto] `compute_hessian`: 2 X^T X + 1e-4 I (no 1/n)."""
    X = np.asarray(X, F64)
    return 2.0 * (X.T @ X) + 1e-4 * np.eye(X.shape[1])


def auto_gptq_quantize_row(weights, H_inv, n_bits: int = 4, group_size: int = 128):
    """[auto] `gptq_quantize_row`: one row, asymmetric group quantizer, static update
    -e / Hinv[c, c] * Hinv[c+1:, c] (skipped when Hinv[c, c] <= 1e-10).
    Returns (codes, [(scale, zero) per group])."""
    w = np.array(weights, dtype=F64, copy=True)
    d = w.shape[0]
    Hinv = np.asarray(H_inv, F64)
    maxq = maxq_asym(n_bits)
    codes = np.zeros(d, dtype=np.int64)
    params = []
    for col in range(d):
        gi = col // group_size
        g0 = gi * group_size
        if col == g0:
            s, z = asym_params(w[None, g0:min(g0 + group_size, d)], maxq, scale_dtype=None)
            params.append((float(s[0]), int(z[0])))
        s, z = params[gi]
        c = int(quant_codes(w[col:col + 1], s, z, n_bits, sym=False)[0])
        codes[col] = c
        err = w[col] - float(dequant(c, s, z, sym=False))
        if col < d - 1 and Hinv[col, col] > 1e-10:
            w[col + 1:] += -err / Hinv[col, col] * Hinv[col + 1:, col]
    return codes, params


def auto_dequantize_row(codes, params, group_size: int = 128) -> np.ndarray:
    codes = np.asarray(codes)
    out = np.zeros(codes.shape[0])
    for col in range(codes.shape[0]):
        s, z = params[col // group_size]
        out[col] = s * (codes[col] - z)
    return out


# ----------------------------------------------------------------------------------------
# comparison helpers used by the parity tests
# ----------------------------------------------------------------------------------------

def perm_equivalent(perm_a, perm_b, keys, rel_tol: float) -> bool:
    """True if two descending orders of `keys` differ only by swaps of keys within
    `rel_tol` of each other (both sort the keys, up to near-ties)."""
    keys = np.asarray(keys, F64)
    a = keys[np.asarray(perm_a)]
    b = keys[np.asarray(perm_b)]
    if sorted(np.asarray(perm_a).tolist()) != list(range(len(keys))):
        return False
    if sorted(np.asarray(perm_b).tolist()) != list(range(len(keys))):
        return False
    scale = np.maximum(np.abs(a), np.abs(b))
    return bool(np.all(np.abs(a - b) <= rel_tol * np.maximum(scale, 1e-300)))
