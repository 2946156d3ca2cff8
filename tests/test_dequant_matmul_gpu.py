"""The consumer of the stored form: gptq_dequant_matmul against the oracle.

Error bound (derived from the arithmetic): every weight is rounded once to bf16 (relative
error <= 2^-9) and the products X[t][k] * Wq_bf16[o][k] are accumulated in fp32 over K
(error <= K * 2^-23 of sum |x w|, rounding or truncating), so elementwise
    |Y_gpu - Y_ref| <= (2^-9 + K * 2^-23) * sum_k |X[t][k]| |Wq[o][k]|.
With scales that are powers of two and small codes the bf16 weights are exact and only
the fp32 accumulation term remains: any wrong code, group, zero point or tile position
fails that tighter bound.
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


def _stored(rng, N, K, bits, G, act, exact):
    u = rng.integers(0, 2 ** bits, size=(N, K))
    if exact:
        scales = 2.0 ** rng.integers(-6, -2, size=(N, G))
    else:
        scales = rng.uniform(0.005, 0.05, size=(N, G))
    scales = scales.astype(np.float32)
    zeros = rng.integers(0, 2 ** bits, size=(N, G)).astype(np.uint8)
    if act:
        g_idx = rng.permutation(np.arange(K) * G // K)       # scattered groups (act_order)
    else:
        g_idx = np.arange(K) * G // K                        # contiguous groups
    return u, scales, zeros, g_idx.astype(np.int32)


def _run(lib, X, u, scales, zeros, g_idx, bits):
    packed = O.pack_rows(u, bits).view(np.int32)
    Y = lib.gptq_dequant_matmul(X, torch.tensor(packed, device=DEV), torch.tensor(scales, device=DEV),
                                torch.tensor(zeros, device=DEV), torch.tensor(g_idx, device=DEV), bits)
    torch.cuda.synchronize()
    return npy(Y).astype(np.float64)


CASES = [
    # T, K, N, bits, G, act_order
    (128, 256, 128, 4, 2, False),
    (300, 320, 200, 3, 5, True),      # ragged tokens and outputs, 5 K steps
    (77, 768, 384, 2, 6, True),
    (513, 1024, 260, 4, 8, False),
    (64, 128, 1000, 3, 1, False),     # one scale per row
]


@pytest.mark.parametrize("T,K,N,bits,G,act", CASES)
@pytest.mark.parametrize("exact", [True, False])
def test_dequant_matmul_matches_oracle(lib, T, K, N, bits, G, act, exact):
    rng = np.random.default_rng(T + K + N + bits + (7 if exact else 0))
    u, scales, zeros, g_idx = _stored(rng, N, K, bits, G, act, exact)
    X = torch.randn(T, K, generator=torch.Generator().manual_seed(T * 31 + K)).to(torch.bfloat16).to(DEV)
    Xh = synth.to_numpy_f64(X)
    Yg = _run(lib, X, u, scales, zeros, g_idx, bits)
    W = O.dequant_stored(O.pack_rows(u, bits), scales.astype(np.float64), zeros, g_idx, bits, K)
    Yr = Xh @ W.T
    mag = np.abs(Xh) @ np.abs(W).T
    acc = K * 2.0 ** -23   # fp32 accumulation, round or truncate
    bound = (acc if exact else 2.0 ** -9 + acc) * mag + 1e-30
    assert np.all(np.abs(Yg - Yr) <= bound), float(np.max(np.abs(Yg - Yr) / bound))


def test_dequant_matmul_consumes_gptq_quantize_output(lib):
    """The stored form gptq_quantize writes (act_order, groups, asymmetric) read back by the
    consumer equals X Wq^T with the loop's own dequantised weights Wq, within the bf16 bound."""
    rng = np.random.default_rng(11)
    K, N = 384, 96
    spec = synth.XSpec(n=2048, d=K, kind="scaled", dtype="bf16", n_outliers=4, outlier_factor=20.0,
                       dead_frac=0.02, segment=1024)
    Xc = synth.make_x(spec, 12, device=DEV)
    h = lib.Hessian(K)
    h.accumulate(Xc)
    H, diag, _ = h.finalize()
    U, perm, dead = lib.gptq_prepare(H, diag, 0.01, act_order=True)
    W = synth.make_weight(N, K, 0.02, 13, device=DEV)
    out = lib.gptq_quantize(W, U, perm, dead, 3, 64, False)
    X = Xc[:200].contiguous()
    Y = lib.gptq_dequant_matmul(X, out["packed"], out["scales"], out["zeros"], out["g_idx"], 3)
    torch.cuda.synchronize()
    Xh = synth.to_numpy_f64(X)
    Wq = npy(out["Wq"]).astype(np.float64)
    Yr = Xh @ Wq.T
    bound = (2.0 ** -9 + K * 2.0 ** -23) * (np.abs(Xh) @ np.abs(Wq).T) + 1e-30
    assert np.all(np.abs(npy(Y).astype(np.float64) - Yr) <= bound)
    del rng


def test_dequant_matmul_rejects_out_of_range_groups(lib):
    rng = np.random.default_rng(3)
    u, scales, zeros, g_idx = _stored(rng, 64, 128, 4, 2, False, True)
    g_idx[5] = 7    # no such group: the kernel records INVALID_ARG and reads group 0
    X = torch.randn(16, 128).to(torch.bfloat16).to(DEV)
    with pytest.raises(lib.GptqError) as e:
        _run(lib, X, u, scales, zeros, g_idx, 4)
    assert e.value.status == 1
