"""Activation quantisation at its rounding boundaries, on every kernel that
quantises, against the oracle.

The quantisation of BitNet 深度拆解 §2.2 rounds fl(fl(x / s) * 127) to the
nearest integer, ties to even.  The kernels take a multiply by fl(127 / s)
first and fall back to the IEEE division only for elements whose product
lies within 2^-14 of a half-integer, so these rows put every element there:
x = fl((k + 1/2) * s / 127) for k = -127 .. 126 and its neighbours up to
three ulps away, with the row's absmax fixed at s (or below 1e-8, where the
scale is the 1e-8 floor).  x_q and the scales must equal the oracle's bit
for bit, and the fused BitLinear's int32 accumulators its contraction.
"""
import numpy as np
import pytest

from test_gpu_parity import to_dev
from ternary_weight_05_b300 import synth

# absmax values of the rows; 5e-9 is below the 1e-8 floor of the scale
AMAX = [1.0, 3.7, 0.0123, 300.0, 5e-9]


def tie_rows(M, K, seed):
    """[M, K] fp32, row m with absmax AMAX[m % len(AMAX)]: half-integer
    products and their neighbours, shuffled, the absmax at a random place."""
    rng = np.random.default_rng(seed)
    rows = np.empty((M, K), dtype=np.float32)
    k = np.arange(-127, 127, dtype=np.float64)
    for m in range(M):
        a = np.float32(AMAX[m % len(AMAX)])
        s = max(float(a), 1e-8)
        base = ((k + 0.5) * (s / 127.0)).astype(np.float32)
        cands = [base]
        up, dn = base, base
        for _ in range(3):
            up = np.nextafter(up, np.float32(np.inf))
            dn = np.nextafter(dn, np.float32(-np.inf))
            cands += [up, dn]
        pool = np.concatenate(cands)
        pool = pool[np.abs(pool) <= a]
        row = rng.choice(pool, size=K)
        row[rng.integers(K)] = a if rng.random() < 0.5 else -a
        rows[m] = row
    return rows


def check_quant(lib, oracle_mod, dev, x_h):
    xq, s = lib.quant_act(to_dev(x_h, dev))
    xq_ref, s_ref = oracle_mod.quant_act(x_h)
    assert np.array_equal(s.cpu().numpy(), s_ref)
    assert np.array_equal(xq.cpu().numpy(), xq_ref)


# K = 2560: rows held in registers; K = 20480: the two-pass loop
@pytest.mark.gpu
@pytest.mark.parametrize("M,K", [(5, 2560), (5, 20480)])
def test_quant_act_at_ties(lib, oracle_mod, cuda_dev, M, K):
    check_quant(lib, oracle_mod, cuda_dev, tie_rows(M, K, seed=M + K))


# the fused BitLinear's quantisation: streaming kernel (1 and 2 tokens),
# row-range kernel (one token, K = 16384), tensor-core prep (5 and 300 tokens)
@pytest.mark.gpu
@pytest.mark.parametrize("M,K", [(1, 2560), (2, 2560), (1, 16384), (5, 2560), (300, 2560)])
def test_bitlinear_quantisation_at_ties(lib, oracle_mod, cuda_dev, M, K):
    N = 96
    W = synth.weights_np(N, K, "normal", 0.02, seed=K + 3)
    x_h = tie_rows(M, K, seed=7 * M + K)
    packed, beta, _ = lib.pack_weights(to_dev(W, cuda_dev))
    y, acc, xq, s = lib.bitlinear(to_dev(x_h, cuda_dev), packed, beta, N, K, want_acc=True, want_xq=True)
    p_ref, b_ref, _ = oracle_mod.pack_weights(W)
    _, acc_ref, xq_ref, s_ref = oracle_mod.bitlinear(x_h, p_ref, b_ref, N, K)
    assert np.array_equal(s.cpu().numpy(), s_ref)
    assert np.array_equal(xq.cpu().numpy(), xq_ref)
    assert np.array_equal(acc.cpu().numpy(), acc_ref)
    lib.check_device_error()


def test_tie_rows_hit_the_boundaries():
    """The rows really sit at the rounding boundaries: in fp64, most products
    x * 127 / s lie within 2^-14 of a half-integer."""
    x = tie_rows(5, 2560, seed=1)
    for m in range(5):
        s = max(float(np.max(np.abs(x[m]))), 1e-8)
        t = x[m].astype(np.float64) * 127.0 / s
        near = np.abs(np.abs(t - np.round(t)) - 0.5) < 2.0 ** -14
        assert near.mean() > 0.9, m
