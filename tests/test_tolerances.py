"""The fp32 tolerances the GPU parity tests use, checked against the exact
values on the CPU by emulating the kernels' fp32 operation sequences with
numpy float32 (each operation rounded once), so that the bounds written in
the tests are shown to hold with margin (and the tests are not flaky)."""
import numpy as np

U = 2.0 ** -24


def f32(x):
    return np.asarray(x, dtype=np.float32)


def test_bitlinear_output_bound():
    # y = fl(acc * fl(fl(beta * s) / 127)): three roundings, < 2^-22 relative,
    # far inside the 1e-6 of the parity tests
    rng = np.random.default_rng(1)
    n = 200000
    K = 8192
    acc = rng.integers(-127 * K, 127 * K, n).astype(np.int64)
    beta = f32(rng.integers(1, 1 << 20, n) / float(1 << 20))
    s = f32(np.abs(rng.standard_normal(n)) * 10 + 1e-3)
    f = f32(f32(beta * s) / f32(127.0))
    y = f32(f32(acc.astype(np.float32)) * f)  # |acc| < 2^24: exact in fp32
    exact = acc.astype(np.float64) * beta.astype(np.float64) * s.astype(np.float64) / 127.0
    nz = exact != 0
    rel = np.abs(y[nz] - exact[nz]) / np.abs(exact[nz])
    assert rel.max() < 2 ** -22
    assert rel.max() < 1e-6


def test_swiglu_bound():
    # fl(fl(yg / fl(1 + exp(-yg))) * yu) with yg, yu each within 3u: the
    # parity tests allow (16 + 4 |yg|) u relative (derivation in the test
    # module); here exp is numpy's float32 exp (within 1 ulp)
    rng = np.random.default_rng(2)
    n = 400000
    yg64 = rng.standard_normal(n) * 6.0
    yu64 = rng.standard_normal(n) * 3.0
    # y's as the kernels form them: the exact value times (1 + up to 3u)
    yg = f32(yg64 * (1 + rng.uniform(-3, 3, n) * U))
    yu = f32(yu64 * (1 + rng.uniform(-3, 3, n) * U))
    e = np.exp(-yg).astype(np.float32)
    a = f32(f32(yg / f32(f32(1.0) + e)) * yu)
    exact = yg64 / (1.0 + np.exp(-yg64)) * yu64
    tol = (16.0 + 4.0 * np.abs(yg64)) * U * np.abs(exact) + 1e-30
    assert np.all(np.abs(a.astype(np.float64) - exact) <= tol)


def _fma32(a, b, c):
    return f32(a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64))


def test_grouped_sum_bound():
    # F = sum_g acc_g * w_g in fp32: per-lane fused multiply-adds over at
    # most 4 groups, then a 5-level butterfly; or sequential fused
    # multiply-adds over all groups; y = fl(F * fl(s / 127)).  The parity
    # tests allow (K/G + 8) u * cond, cond = (s/127) sum_g |acc_g w_g|.
    rng = np.random.default_rng(3)
    for ng in (2, 16, 64, 128):
        trials = 3000
        acc = rng.integers(-127 * 128, 127 * 128, (trials, ng)).astype(np.float32)
        w = f32(rng.standard_normal((trials, ng)) * 0.05)
        s = f32(np.abs(rng.standard_normal(trials)) + 0.1)
        t = f32(s / f32(127.0))
        # order 1: sequential FMA
        F1 = np.zeros(trials, dtype=np.float32)
        for g in range(ng):
            F1 = _fma32(acc[:, g], w[:, g], F1)
        # order 2: 32 lanes, lane l holding groups l, l + 32, ... then a butterfly
        lanes = np.zeros((trials, 32), dtype=np.float32)
        for g in range(ng):
            lanes[:, g % 32] = _fma32(acc[:, g], w[:, g], lanes[:, g % 32])
        for o in (16, 8, 4, 2, 1):
            lanes = f32(lanes + lanes[:, np.arange(32) ^ o])
        F2 = lanes[:, 0]
        exact = (acc.astype(np.float64) * w.astype(np.float64)).sum(axis=1) * s.astype(np.float64) / 127.0
        cond = np.abs(acc.astype(np.float64) * w.astype(np.float64)).sum(axis=1) * s.astype(np.float64) / 127.0
        for F in (F1, F2):
            y = f32(F * t).astype(np.float64)
            assert np.all(np.abs(y - exact) <= (ng + 8) * U * cond)
