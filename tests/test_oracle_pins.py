"""Pins the CPU oracle to what the pages and mathematics fix (no GPU).

Each test states the fact it checks.  None of them re-types the oracle's own
formula: they use hand-derived worked examples (tests/golden), invariants,
closed forms, exact rational arithmetic, brute force on tiny inputs, and the
alternative formulations the pages give.
"""
import itertools
import math
from fractions import Fraction

import numpy as np
import pytest

from conftest import load_golden

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ---------------------------------------------------------------- packing ---

def test_pack_worked_tuples(oracle_mod):
    g = load_golden("pack_tuples.json")
    for case in g["cases"]:
        got = oracle_mod.pack_codes(np.array(case["ternary"], dtype=np.int8))
        assert got.tolist() == case["packed"], case


def test_pack_all_81_tuples_round_trip_and_bijection(oracle_mod):
    # 3^4 ternary 4-tuples: each packs to one byte, unpacking returns it, the 81
    # bytes are distinct and no 2-bit field is 3 (codes are w+1 in {0,1,2}).
    tuples = np.array(list(itertools.product([-1, 0, 1], repeat=4)), dtype=np.int8)
    packed = oracle_mod.pack_codes(tuples.ravel())
    assert packed.size == 81  # four weights per byte
    assert len(set(packed.tolist())) == 81
    for b in packed.tolist():
        assert all(((b >> (2 * s)) & 3) != 3 for s in range(4))
    back = oracle_mod.unpack_codes(packed, tuples.size)
    assert np.array_equal(back, tuples.ravel())


def test_pack_round_trip_random_and_sizes(oracle_mod):
    rng = np.random.default_rng(7)
    for n in [1, 2, 3, 4, 5, 7, 8, 1023, 4096, 4097]:
        q = rng.integers(-1, 2, size=n).astype(np.int8)
        p = oracle_mod.pack_codes(q)
        assert p.size == (n + 3) // 4
        assert np.array_equal(oracle_mod.unpack_codes(p, n), q)
        # ragged tail: padding fields hold code 0
        if n % 4:
            last = int(p[-1])
            for s in range(n % 4, 4):
                assert (last >> (2 * s)) & 3 == 0


def test_unpack_reads_code3_as_plus2(oracle_mod):
    # unpack_ternary subtracts 1 from the raw field; a field 3 (never produced
    # by packing) therefore reads +2.
    assert oracle_mod.unpack_codes(np.array([0xFF], dtype=np.uint8), 4).tolist() == [2, 2, 2, 2]


# ---------------------------------------------------------- ternarisation ---

def _check_pack_golden(oracle_mod, name):
    g = load_golden(name)
    W = np.array(g["W"], dtype=np.float32)
    packed, beta, am = oracle_mod.pack_weights(W)
    assert packed.tolist() == g["packed"]
    assert float(beta) == g["beta"]
    n = W.size
    assert oracle_mod.unpack_codes(packed, n).tolist() == g["ternary"]
    if "absmean" in g:
        assert float(am) == g["absmean"]
        assert float(oracle_mod.gamma(am)) == g["gamma"]


def test_ternarize_worked_example_round_half_even_and_clamp(oracle_mod):
    _check_pack_golden(oracle_mod, "ternarize_worked.json")


def test_ternarize_multiplies_by_reciprocal(oracle_mod):
    _check_pack_golden(oracle_mod, "ternarize_reciprocal.json")


def test_ternarize_thresholds_at_half_gamma(oracle_mod):
    # With gamma = 1 (mean|W| = 1), the code is the nearest integer clamped to
    # [-1, 1]: |w| < 0.5 -> 0, |w| > 0.5 -> sign(w); exact halves go to 0.
    for w, want in [(0.4999, 0), (0.5001, 1), (-0.5001, -1), (7.0, 1), (-7.0, -1), (0.0, 0),
                    (-0.0, 0), (1e-30, 0), (np.inf, 1), (-np.inf, -1)]:
        assert oracle_mod.ternarize(1.0, w) == want, w


@pytest.mark.parametrize("R", [4.0, 0.05, 300.0])
def test_pack_every_bf16_weight_like_the_page_listing(oracle_mod, R):
    # Every finite bf16 weight with |w| <= R in one matrix (so mean|W|, and
    # with it gamma, differ per R): the oracle's codes equal the absmean
    # listing of BitNet 深度拆解 section 2.2 run in torch CPU fp32 on the same
    # mean (gamma = 1 / (alpha * mean + eps), clamp(round(gamma * w), -1, 1)),
    # and beta is the listing's mean(|W_ternary|).
    import torch

    v = _all_finite_bf16()
    v = v[np.abs(v) <= R]
    n = v.size - v.size % 4
    W = v[:n].reshape(4, n // 4).astype(np.float32)
    packed, beta, am = oracle_mod.pack_weights(W)
    Wt = torch.from_numpy(W)
    gamma = 1.0 / (1.0 * torch.tensor(am, dtype=torch.float32) + 1e-8)
    wt = torch.clamp(torch.round(gamma * Wt), -1, 1)
    assert np.array_equal(oracle_mod.unpack_codes(packed, W.size), wt.numpy().astype(np.int8).ravel())
    assert beta == np.float32(float(wt.abs().mean(dtype=torch.float64)))  # nnz / n, rounded once
    # and codes of both signs and zeros occur
    assert {-1, 0, 1} <= set(np.unique(wt.numpy()).astype(int).tolist())


def test_absmean_equals_exact_mean_to_fp32_rounding(oracle_mod):
    rng = np.random.default_rng(3)
    for n in [1, 5, 4095, 4096, 4097, 20000]:
        w = (rng.standard_normal(n) * rng.choice([1e-3, 1.0, 50.0])).astype(np.float32)
        exact = sum(Fraction(float(abs(v))) for v in w) / n
        got = oracle_mod.absmean(w)
        # fp64 accumulation error is far below half an fp32 ulp, so the result
        # is within one fp32 ulp of the exact mean (and almost always equal to
        # the correctly rounded value).
        ulp = np.spacing(np.float32(float(exact)))
        assert abs(Fraction(float(got)) - exact) <= Fraction(float(ulp))
        assert got == np.float32(float(exact)) or n > 4096


def test_gamma_special_cases(oracle_mod):
    # mean 1 -> gamma exactly 1 (eps vanishes in fp32); mean 0 (all-zero
    # weights) -> gamma = 1/fl32(1e-8); alpha scales the mean.
    assert float(oracle_mod.gamma(1.0)) == 1.0
    assert float(oracle_mod.gamma(0.0)) == float(np.float32(1.0) / np.float32(1e-8))
    assert float(oracle_mod.gamma(2.0, alpha=0.5)) == 1.0
    assert float(oracle_mod.gamma(0.25)) == 4.0


def test_all_zero_weights_give_beta_zero_and_zero_output(oracle_mod):
    # An all-zero weight matrix (a checkpoint defect reported in the
    # microsoft-bitnet review, section 06) must ternarise to all zeros.
    W = np.zeros((8, 16), dtype=np.float32)
    packed, beta, am = oracle_mod.pack_weights(W)
    assert float(beta) == 0.0 and float(am) == 0.0
    assert np.all(packed == 0x55)  # every code is 1 (weight 0)
    x = np.random.default_rng(0).standard_normal((3, 16)).astype(np.float32)
    y, acc, _, _ = oracle_mod.bitlinear(x, packed, beta, 8, 16)
    assert np.all(acc == 0) and np.all(y == 0)


def _phi(z):
    return 0.5 * (1.0 + math.erf(z / math.sqrt(2.0)))


@pytest.mark.parametrize("dist", ["gauss", "laplace"])
def test_beta_closed_form(oracle_mod, dist):
    # For i.i.d. W, gamma ~ 1/E|W| and P(code 0) = P(|W| < E|W|/2):
    #   Gaussian: E|W| = sigma*sqrt(2/pi), P0 = 2*Phi(sqrt(2/pi)/2) - 1 = 0.3101
    #   Laplace(b): E|W| = b, P0 = 1 - exp(-1/2) = 0.3935
    # beta = 1 - P0 must hold within binomial noise (5 sigma).
    rng = np.random.default_rng(11)
    N, K = 1024, 2048
    if dist == "gauss":
        W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
        p0 = 2 * _phi(math.sqrt(2 / math.pi) / 2) - 1
    else:
        W = rng.laplace(0.0, 0.01, (N, K)).astype(np.float32)
        p0 = 1 - math.exp(-0.5)
    _, beta, _ = oracle_mod.pack_weights(W)
    n = N * K
    sigma = math.sqrt(p0 * (1 - p0) / n)
    assert abs(float(beta) - (1 - p0)) < 5 * sigma + 2e-4


# --------------------------------------------------------- quant_act ---

def test_quant_act_worked_example(oracle_mod):
    g = load_golden("quant_act_worked.json")
    xq, s = oracle_mod.quant_act(np.array(g["x"], dtype=np.float32))
    assert xq.tolist() == g["x_q"]
    assert [float(v) for v in s] == [float(np.float32(v)) for v in g["scale"]]


def _all_finite_bf16():
    bits = np.arange(1 << 16, dtype=np.uint32)
    f = (bits << 16).view(np.float32)
    return f[np.isfinite(f)]


@pytest.mark.parametrize("smax", [1.0, 3.0, 0.0123, 1000.0])
def test_quant_act_all_bf16_within_half_step(oracle_mod, smax):
    # Every finite bf16 value v with |v| <= smax, placed in a row whose absmax
    # is smax, must quantise to the integer nearest 127*v/smax (the exact real
    # value), up to the fp32 rounding of the two operations (< 4e-5), with
    # the row maximum mapping to exactly 127.
    v = _all_finite_bf16()
    v = v[np.abs(v) <= smax]
    x = np.zeros((v.size, 2), dtype=np.float32)
    x[:, 0] = smax
    x[:, 1] = v
    xq, s = oracle_mod.quant_act(x)
    assert np.all(s == np.float32(smax))
    assert np.all(xq[:, 0] == 127)
    exact = 127.0 * v.astype(np.float64) / np.float64(np.float32(smax))
    assert np.all(np.abs(xq[:, 1] - exact) <= 0.5 + 4e-5)
    # sign preserved, monotone in v
    assert np.all(np.sign(xq[:, 1]) * np.sign(v) >= 0)
    order = np.argsort(v, kind="stable")
    assert np.all(np.diff(xq[order, 1].astype(np.int32)) >= 0)


def test_quant_act_divides_first_like_the_page_listing(oracle_mod):
    # fp32 rows whose absmax is the first element and whose other elements
    # round to different codes under fl(fl(x / s) * 127) and fl(x * fl(127 /
    # s)): the absmax_quantize listing of BitNet 深度拆解 section 2.2
    # (torch.round(x / scales * qmax), run in torch CPU fp32) decides
    import torch

    rows = [[3.3, 3.235039472579956, 1.8578739166259766],
            [0.7071, 0.6319357752799988, -0.4314979910850525, 0.6876129508018494, 0.2978728115558624],
            [5.123, 3.933011770248413]]
    for r in rows:
        x = np.array([r], np.float32)
        xq, s = oracle_mod.quant_act(x)
        xt = torch.from_numpy(x)
        scales = xt.abs().amax(dim=-1, keepdim=True).clamp_min(1e-8)
        ref = torch.clamp(torch.round(xt / scales * 127), -127, 127)
        assert np.array_equal(xq, ref.numpy().astype(np.int8))
        # the rows do tell the two orders apart
        other = np.rint(x * np.float32(np.float32(127.0) / s[0])).astype(np.int8)
        assert not np.array_equal(other, xq)


def test_quant_act_invariants(oracle_mod):
    rng = np.random.default_rng(5)
    x = (rng.standard_t(4, size=(64, 777)) * rng.choice([1e-6, 1.0, 1e4])).astype(np.float32)
    x[3] = 0.0
    xq, s = oracle_mod.quant_act(x)
    assert np.all(np.abs(xq.astype(np.int32)) <= 127)  # -128 never produced
    assert np.all(s[np.arange(64) != 3] == np.abs(x[np.arange(64) != 3]).max(axis=1))
    assert s[3] == np.float32(1e-8) and np.all(xq[3] == 0)
    # the element holding the row absmax maps to exactly +/-127
    idx = np.abs(x).argmax(axis=1)
    for m in range(64):
        if m != 3:
            assert abs(int(xq[m, idx[m]])) == 127


# ------------------------------------------------------- contraction ---

def test_contraction_worked_example(oracle_mod):
    g = load_golden("bitlinear_worked.json")
    xq = np.array(g["x_q"], dtype=np.int8)
    acc = oracle_mod.contract(xq, np.array(g["packed"], dtype=np.uint8), g["N"], g["K"])
    assert acc.tolist() == g["acc"]
    y = oracle_mod.epilogue(acc, np.array(g["scale"], dtype=np.float32), g["beta"])
    assert y.tolist() == g["y"]


def test_contraction_ternary_product_identity(oracle_mod):
    # -1*x = -x, 0*x = 0, +1*x = x (BitNet 深度拆解 section 1): with a one-hot
    # activation v*e_k, acc[n] equals (w[n,k]) * v exactly.
    rng = np.random.default_rng(9)
    N, K = 6, 12
    q = rng.integers(-1, 2, size=(N, K)).astype(np.int8)
    packed = oracle_mod.pack_codes(q)
    for k in range(K):
        for v in (-127, -1, 1, 77, 127):
            x = np.zeros((1, K), dtype=np.int8)
            x[0, k] = v
            acc = oracle_mod.contract(x, packed, N, K)
            assert acc[0].tolist() == [int(q[n, k]) * v for n in range(N)]


@pytest.mark.parametrize("M,N,K", [(1, 1, 4), (3, 5, 8), (4, 7, 20), (2, 9, 100)])
def test_contraction_equals_fp64_matmul(oracle_mod, M, N, K):
    # A float64 matmul of the unpacked ternary matrix with x_q is exact for
    # these magnitudes and must equal the integer accumulator.
    rng = np.random.default_rng(M * 100 + N * 10 + K)
    q = rng.integers(-1, 2, size=(N, K)).astype(np.int8)
    xq = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    acc = oracle_mod.contract(xq, oracle_mod.pack_codes(q), N, K)
    ref = xq.astype(np.float64) @ q.astype(np.float64).T
    assert np.array_equal(acc.astype(np.float64), ref)


def test_contraction_equals_sign_mask_loop(oracle_mod):
    # The sign/mask loop of the devpress post ("三值量化：把乘法变成加减法"):
    # acc += x if sign > 0 else -x wherever the nonzero mask is set.
    rng = np.random.default_rng(21)
    N, K = 5, 16
    q = rng.integers(-1, 2, size=(N, K)).astype(np.int8)
    x = rng.integers(-127, 128, size=(1, K)).astype(np.int8)
    sign = np.where(q >= 0, 1, -1)
    mask = q != 0
    out = []
    for o in range(N):
        a = 0
        for i in range(K):
            if mask[o, i]:
                a += int(x[0, i]) if sign[o, i] > 0 else -int(x[0, i])
        out.append(a)
    acc = oracle_mod.contract(x, oracle_mod.pack_codes(q), N, K)
    assert acc[0].tolist() == out


def test_contraction_row_ranges_and_threads(oracle_mod):
    rng = np.random.default_rng(2)
    N, K, M = 37, 64, 3
    q = rng.integers(-1, 2, size=(N, K)).astype(np.int8)
    xq = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    p = oracle_mod.pack_codes(q)
    full = oracle_mod.contract(xq, p, N, K)
    assert np.array_equal(oracle_mod.contract(xq, p, N, K, threads=4), full)
    part = oracle_mod.contract(xq, p, N, K, rows=(10, 20))
    assert np.array_equal(part[:, 10:20], full[:, 10:20])
    assert np.all(part[:, :10] == 0) and np.all(part[:, 20:] == 0)


# ---------------------------------------------------------- epilogue ---

def test_epilogue_matches_exact_rational(oracle_mod):
    # y = acc * beta * s / 127 computed exactly with rationals, then rounded to
    # the nearest fp32: the oracle is within half an fp32 ulp (plus the tiny
    # fp64 error before the final rounding).
    rng = np.random.default_rng(4)
    M, N = 7, 33
    acc = rng.integers(-2_000_000, 2_000_000, size=(M, N)).astype(np.int32)
    acc[0, 0] = 0
    s = (rng.random(M) * 10 + 1e-8).astype(np.float32)
    beta = np.float32(0.6899)
    y = oracle_mod.epilogue(acc, s, float(beta))
    for m in range(M):
        for n in range(N):
            exact = Fraction(int(acc[m, n])) * Fraction(float(beta)) * Fraction(float(s[m])) / 127
            got = Fraction(float(y[m, n]))
            if exact == 0:
                assert got == 0
                continue
            ulp = Fraction(float(np.spacing(np.float32(abs(float(exact))))))
            assert abs(got - exact) <= ulp / 2 + abs(exact) * Fraction(1, 10**12)


def test_epilogue_zero_beta(oracle_mod):
    acc = np.array([[5, -7]], dtype=np.int32)
    assert oracle_mod.epilogue(acc, np.array([3.0], np.float32), 0.0).tolist() == [[0.0, 0.0]]


# --------------------------------------------- whole BitLinear forward ---

def test_bitlinear_forward_matches_page_torch_formulation(oracle_mod):
    # The BitLinear forward of BitNet 深度拆解 section 3.1, run through torch CPU:
    # F.linear of the integer-valued fp32 operands is exact (|acc| < 2^24), and
    # the rescale (with weight_scale = beta and act_scale = absmax/127) agrees
    # with the oracle to fp32 rounding.
    import torch
    import torch.nn.functional as F

    rng = np.random.default_rng(12)
    M, N, K = 4, 96, 256
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    x = rng.standard_normal((M, K)).astype(np.float32)
    packed, beta, _ = oracle_mod.pack_weights(W)
    y, acc, xq, s = oracle_mod.bitlinear(x, packed, beta, N, K)
    wt = torch.from_numpy(oracle_mod.unpack_codes(packed, N * K).reshape(N, K).astype(np.float32))
    out_q = F.linear(torch.from_numpy(xq.astype(np.float32)), wt)
    assert np.array_equal(out_q.numpy(), acc.astype(np.float32))
    ref = (out_q.double() * float(beta) * torch.from_numpy(s).double()[:, None] / 127.0).float()
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-6, atol=0)
    # gamma from torch's own mean agrees with the fixed-order mean here
    tmean = torch.from_numpy(W).abs().mean()
    tq = torch.clamp(torch.round((1.0 / (1.0 * tmean + 1e-8)) * torch.from_numpy(W)), -1, 1)
    assert np.array_equal(tq.numpy().astype(np.int8), wt.numpy().astype(np.int8))


# ------------------------------------------------ SwiGLU (FFN, next row) ---

def test_silu_special_values(oracle_mod):
    # sigmoid(ln 3) = 1 / (1 + 1/3) = 3/4, so silu(+-ln 3) = +-ln 3 * {3/4, 1/4}:
    # a dropped minus sign in exp(-z) swaps the two values
    ln3 = np.log(3.0)
    assert oracle_mod.silu(ln3) == pytest.approx(0.75 * ln3, rel=1e-15)
    assert oracle_mod.silu(-ln3) == pytest.approx(-0.25 * ln3, rel=1e-15)
    assert oracle_mod.silu(0.0) == 0.0
    assert oracle_mod.silu(60.0) == 60.0  # sigmoid rounds to 1
    assert -1e-20 < oracle_mod.silu(-60.0) < 0.0


def test_silu_odd_part_is_identity(oracle_mod):
    # silu(z) - silu(-z) = z (sigmoid(z) + sigmoid(-z) = 1)
    for z in np.linspace(-30.0, 30.0, 241):
        assert oracle_mod.silu(z) - oracle_mod.silu(-z) == pytest.approx(z, abs=1e-12)


def test_swiglu_uses_exact_bitlinear_outputs(oracle_mod):
    # acc * w_scale * s / 127 with s = 127, w_scale = 1 is the accumulator itself
    acc_g = np.array([[0, 3, -3, 40]], dtype=np.int32)
    acc_u = np.array([[5, 2, 2, -1]], dtype=np.int32)
    out = oracle_mod.swiglu(acc_g, acc_u, np.array([127.0], np.float32), 1.0, 1.0)
    expect = [0.0, 2 * oracle_mod.silu(3.0), 2 * oracle_mod.silu(-3.0), -oracle_mod.silu(40.0)]
    assert np.allclose(out[0], expect, rtol=1e-15, atol=0)
    # gate and up scales enter separately
    out2 = oracle_mod.swiglu(acc_g, acc_u, np.array([127.0], np.float32), 0.5, 2.0)
    assert out2[0, 1] == pytest.approx(oracle_mod.silu(1.5) * 4.0, rel=1e-15)


def test_bitlinear_swiglu_matches_two_bitlinears(oracle_mod):
    rng = np.random.default_rng(3)
    I, K = 20, 64
    Wg = rng.normal(0, 0.02, (I, K)).astype(np.float32)
    Wu = rng.normal(0, 0.02, (I, K)).astype(np.float32)
    pg, bg, _ = oracle_mod.pack_weights(Wg)
    pu, bu, _ = oracle_mod.pack_weights(Wu)
    x = rng.normal(0, 1, (2, K)).astype(np.float32)
    out, acc_g, acc_u, _, s = oracle_mod.bitlinear_swiglu(x, pg, bg, pu, bu, I, K)
    yg, acc_g2, _, _ = oracle_mod.bitlinear(x, pg, bg, I, K)
    yu, acc_u2, _, _ = oracle_mod.bitlinear(x, pu, bu, I, K)
    assert np.array_equal(acc_g, acc_g2) and np.array_equal(acc_u, acc_u2)
    # the fp32 BitLinear outputs are within one rounding of the exact ones
    ref = np.array([[oracle_mod.silu(float(a)) * float(b) for a, b in zip(ra, rb)] for ra, rb in zip(yg, yu)])
    assert np.allclose(out, ref, rtol=1e-5, atol=1e-12)


# ------------------------------------------------- group-wise weight scales --

def test_grouped_worked_example(oracle_mod):
    g = load_golden("grouped_worked.json")
    W = np.array(g["W"], dtype=np.float32)
    packed, ws, am = oracle_mod.pack_weights_grouped(W, g["G"])
    assert packed.tolist() == g["packed"]
    assert oracle_mod.unpack_codes(packed, W.size).reshape(W.shape).tolist() == g["ternary"]
    assert ws.tolist() == g["w_scale"]
    assert am.tolist() == g["absmean"]
    acc_g = oracle_mod.contract_grouped(np.array(g["x_q"], dtype=np.int8), packed, W.shape[0], W.shape[1], g["G"])
    assert acc_g.tolist() == g["acc_g"]
    y, cond = oracle_mod.epilogue_grouped(acc_g, np.array(g["scale"], dtype=np.float32), ws)
    assert y.tolist() == g["y"] and cond.tolist() == g["cond"]


def test_grouped_groups_are_independent(oracle_mod):
    """Scaling one group's weights by a power of two leaves every code and
    beta unchanged and scales that group's absmean exactly (a global or
    per-row mean would move the thresholds of the other groups)."""
    rng = np.random.default_rng(11)
    N, K, G = 6, 512, 128
    W = rng.standard_normal((N, K)).astype(np.float32) * np.float32(0.02)
    p0, ws0, am0 = oracle_mod.pack_weights_grouped(W, G)
    W2 = W.copy()
    W2[2, G:2 * G] *= np.float32(64.0)
    W2[5, 3 * G:] *= np.float32(0.125)
    p1, ws1, am1 = oracle_mod.pack_weights_grouped(W2, G)
    assert np.array_equal(p0, p1) and np.array_equal(ws0, ws1)
    expect = am0.copy()
    expect[2, 1] *= np.float32(64.0)
    expect[5, 3] *= np.float32(0.125)
    assert np.array_equal(am1, expect)
    # and a per-tensor pack of the modified matrix does change codes
    pt, _, _ = oracle_mod.pack_weights(W2)
    assert not np.array_equal(pt, p1)


def test_grouped_pack_thresholds_per_group(oracle_mod):
    """Within each group, |w| * gamma_g > 1/2 decides a nonzero code (away
    from exact ties), with gamma_g = 1 / (mean|W_g| + eps) from that group
    alone; beta_g counts those codes."""
    rng = np.random.default_rng(12)
    N, K, G = 4, 256, 64
    W = rng.laplace(0.0, 0.01, (N, K)).astype(np.float32)
    packed, ws, am = oracle_mod.pack_weights_grouped(W, G)
    q = oracle_mod.unpack_codes(packed, N * K).reshape(N, K)
    for n in range(N):
        for gi in range(K // G):
            w = W[n, gi * G:(gi + 1) * G].astype(np.float64)
            mean = np.mean(np.abs(w))
            assert abs(am[n, gi] - mean) <= 1e-6 * mean
            t = np.abs(w) / mean
            qq = q[n, gi * G:(gi + 1) * G]
            clear = np.abs(t - 0.5) > 1e-5
            assert np.all((qq[clear] != 0) == (t[clear] > 0.5))
            assert np.all(np.sign(qq) == np.where(qq != 0, np.sign(w), 0))
            assert ws[n, gi] == np.count_nonzero(qq) / G


def test_grouped_one_group_per_row_is_per_channel(oracle_mod):
    """G = K: each row is ternarised on its own; the bytes of row n equal the
    per-tensor pack of the 1 x K matrix W[n] (the per-channel scale)."""
    rng = np.random.default_rng(13)
    N, K = 5, 96
    W = (rng.standard_normal((N, K)) * np.exp(rng.standard_normal((N, 1)))).astype(np.float32)
    packed, ws, am = oracle_mod.pack_weights_grouped(W, K)
    for n in range(N):
        p, b, a = oracle_mod.pack_weights(W[n:n + 1])
        assert np.array_equal(packed[n * K // 4:(n + 1) * K // 4], p)
        assert ws[n, 0] == np.float32(b) and am[n, 0] == np.float32(a)


@pytest.mark.parametrize("M,N,K,G", [(1, 3, 64, 8), (3, 5, 96, 32), (2, 4, 256, 256)])
def test_grouped_matmul_equals_dense_dequantised_fp64(oracle_mod, M, N, K, G):
    """Brute force: y = (x_q * s / 127) @ (W_ternary * w_scale[n, k // G])^T
    with a dense fp64 matmul of the dequantised operands; and the group sums
    add up to the per-tensor integer product."""
    rng = np.random.default_rng(M * 100 + N + K)
    q = rng.integers(-1, 2, size=(N, K)).astype(np.int8)
    packed = oracle_mod.pack_codes(q)
    ws = (rng.random((N, K // G)) + 0.1).astype(np.float32)
    xq = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    s = (rng.random(M) * 3 + 0.1).astype(np.float32)
    acc_g = oracle_mod.contract_grouped(xq, packed, N, K, G)
    assert np.array_equal(acc_g.sum(axis=2), oracle_mod.contract(xq, packed, N, K))
    y, cond = oracle_mod.epilogue_grouped(acc_g, s, ws)
    Wd = q.astype(np.float64) * np.repeat(ws.astype(np.float64), G, axis=1)
    Xd = xq.astype(np.float64) * (s.astype(np.float64)[:, None] / 127.0)
    y_dense = Xd @ Wd.T
    assert np.allclose(y, y_dense, rtol=1e-12, atol=1e-12 * np.abs(y_dense).max())
    assert np.all(cond >= np.abs(y) * (1 - 1e-12))
    # equal scales reduce to the per-tensor epilogue
    ws1 = np.full_like(ws, 0.625)
    y1, _ = oracle_mod.epilogue_grouped(acc_g, s, ws1)
    acc = oracle_mod.contract(xq, packed, N, K)
    assert np.allclose(y1, acc * 0.625 * s.astype(np.float64)[:, None] / 127.0, rtol=1e-14, atol=0)


# ------------------------------------- fake-quant (training) forward, NEXT-4 --

@pytest.mark.parametrize("learned", [False, True])
def test_fake_quant_forward_matches_page_torch_module(oracle_mod, learned):
    """The training BitLinear module of BitNet 深度拆解 section 3.1 written out
    in torch CPU ops (fp32 shadow weight, torch mean for absmean, torch.round,
    F.linear of the integer-valued operands, out * act_scale * weight_scale
    with act_scale = absmax / 127) against the oracle's composition."""
    import torch
    import torch.nn.functional as F

    rng = np.random.default_rng(21 + learned)
    M, N, K = 3, 64, 320
    W = (rng.standard_normal((N, K)) / np.sqrt(K)).astype(np.float32)  # the module's init scale
    x = rng.standard_normal((M, K)).astype(np.float32)
    ws = (rng.standard_normal(N) * 0.5 + 1.0).astype(np.float32) if learned else None
    y, cond, acc, xq, s, packed, beta = oracle_mod.bitlinear_fake_quant(W, x, ws)

    Wt = torch.from_numpy(W)
    gamma = 1.0 / (1.0 * Wt.abs().mean() + 1e-8)
    w_t = torch.clamp(torch.round(Wt * gamma), -1, 1)
    beta_t = w_t.abs().mean()
    xt = torch.from_numpy(x)
    amax = xt.abs().amax(dim=-1, keepdim=True).clamp_min(1e-8)
    x_q = torch.clamp(torch.round(xt / amax * 127), -127, 127)
    out_q = F.linear(x_q, w_t)
    scale_n = torch.from_numpy(ws).double() if learned else beta_t.double()
    ref = out_q.double() * (amax.double() / 127.0) * scale_n

    assert np.array_equal(w_t.numpy().astype(np.int8).ravel(), oracle_mod.unpack_codes(packed, N * K))
    assert float(beta) == float(beta_t)
    assert np.array_equal(x_q.numpy().astype(np.int8), xq)
    assert np.array_equal(out_q.numpy(), acc.astype(np.float32))
    if learned:
        np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=0)
        assert np.all(cond >= np.abs(y) * (1 - 1e-12))
    else:
        np.testing.assert_allclose(y, ref.float().numpy(), rtol=3e-7, atol=0)


# ----------------------------------------- RMSNorm in front of a BitLinear --

def test_rmsnorm_worked_examples(oracle_mod):
    # [3, 4, 0, 0]: mean square 25/4, rms 5/2, h = [6/5, 8/5, 0, 0].  Constant
    # rows normalise to 1: a LayerNorm (x - mean) would give 0, a sum instead
    # of a mean 1/2, a missing square root 1/c.  (In every row eps = 2^-23 is
    # below half an ulp of the mean square, so t = ms.)  The weight multiplies
    # element by element.
    x = np.array([[3, 4, 0, 0], [2, 2, 2, 2], [-5, -5, -5, -5], [6, 6, 6, 6]], np.float32)
    h, ms = oracle_mod.rmsnorm(x)
    assert ms.tolist() == [6.25, 4.0, 25.0, 36.0]
    assert h[0].tolist() == np.array([1.2, 1.6, 0, 0], np.float32).tolist()
    assert h[1:].tolist() == [[1.0] * 4, [-1.0] * 4, [1.0] * 4]
    g = np.array([1, -2, 0.5, 4], np.float32)
    hg, _ = oracle_mod.rmsnorm(x, g)
    assert hg[1:].tolist() == [g.tolist(), (-g).tolist(), g.tolist()]


def test_rmsnorm_eps_enters_under_the_root(oracle_mod):
    # A constant row c = 2^-12: c^2 = 2^-24, t = 2^-24 + 2^-23 = 3 * 2^-24, so
    # h = c / sqrt(3 c^2) = 1/sqrt(3).  eps added to the rms instead would give
    # ~0.9995, a dropped eps 1.
    c = 2.0 ** -12
    h, ms = oracle_mod.rmsnorm(np.full((1, 64), c, np.float32))
    assert ms[0] == np.float32(2.0 ** -24)
    assert np.allclose(h, 1.0 / math.sqrt(3.0), rtol=4 * 2.0 ** -24, atol=0)
    # a zero row stays zero (t = eps > 0): no NaN
    h0, ms0 = oracle_mod.rmsnorm(np.zeros((1, 16), np.float32))
    assert ms0[0] == 0.0 and np.all(h0 == 0.0)


@pytest.mark.parametrize("sigma", [1e-2, 1.0, 300.0])
def test_rmsnorm_output_has_unit_rms(oracle_mod, sigma):
    # mean_k h_k^2 = ms / (ms + eps) up to fp32 rounding of each h_k
    rng = np.random.default_rng(int(sigma * 100))
    x = (rng.standard_normal((3, 4096)) * sigma).astype(np.float32)
    h, ms = oracle_mod.rmsnorm(x)
    eps = oracle_mod.RMS_EPS
    got = (h.astype(np.float64) ** 2).mean(axis=1)
    expect = ms.astype(np.float64) / (ms.astype(np.float64) + eps)
    assert np.allclose(got, expect, rtol=1e-6, atol=0)


def test_rmsnorm_scale_invariant_bitwise(oracle_mod):
    # x -> 2^j x scales the mean square by 4^j exactly; with eps below half an
    # ulp of both mean squares, r scales by 2^-j and h is unchanged bit for bit
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((4, 2560)) * 16).astype(np.float32)
    h, ms = oracle_mod.rmsnorm(x)
    assert ms.min() > 64
    for j in (-2, 3):
        hj, msj = oracle_mod.rmsnorm(x * np.float32(2.0 ** j))
        assert np.array_equal(msj, ms * np.float32(4.0 ** j))
        assert np.array_equal(hj, h)


def test_rmsnorm_permutation_equivariant(oracle_mod):
    # values on a grid of 2^-4 (squares exact, the fp64 sum exact in any
    # order): permuting the columns of x and g permutes the columns of h
    rng = np.random.default_rng(6)
    K = 1024
    x = (rng.integers(-200, 201, size=(3, K)) / 16.0).astype(np.float32)
    g = (rng.integers(1, 64, size=K) / 32.0).astype(np.float32)
    perm = rng.permutation(K)
    h, _ = oracle_mod.rmsnorm(x, g)
    hp, _ = oracle_mod.rmsnorm(x[:, perm], g[perm])
    assert np.array_equal(hp, h[:, perm])


def test_rmsnorm_mean_square_in_fp64(oracle_mod):
    # [2^12, 1, 1, ...]: S = 2^24 + (K - 1) exactly (an fp32 running sum stays
    # at 2^24); ms is S / K rounded to fp32
    K = 1000
    x = np.ones(K, np.float32)
    x[0] = 4096.0
    S = oracle_mod.sum_squares(x)
    assert S == 2.0 ** 24 + K - 1
    _, ms = oracle_mod.rmsnorm(x[None, :])
    exact = Fraction(2 ** 24 + K - 1, K)
    cand = np.float32(float(exact))
    lo, hi = np.nextafter(cand, np.float32(-np.inf)), np.nextafter(cand, np.float32(np.inf))
    best = min((cand, lo, hi), key=lambda v: abs(Fraction(float(v)) - exact))
    assert ms[0] == best


def test_rmsnorm_matches_torch_module(oracle_mod):
    # torch.nn.RMSNorm (the norm of the BitTransformer block) in fp64 with the
    # same eps and weight: the oracle's fp32 h is within its six roundings
    import torch

    rng = np.random.default_rng(8)
    M, K = 5, 2560
    x = (rng.standard_normal((M, K)) * np.exp(rng.standard_normal((M, 1)))).astype(np.float32)
    g = (1.0 + 0.1 * rng.standard_normal(K)).astype(np.float32)
    norm = torch.nn.RMSNorm(K, eps=oracle_mod.RMS_EPS, dtype=torch.float64)
    with torch.no_grad():
        norm.weight.copy_(torch.from_numpy(g.astype(np.float64)))
        ref = norm(torch.from_numpy(x.astype(np.float64))).numpy()
    h, _ = oracle_mod.rmsnorm(x, g)
    assert np.all(np.abs(h - ref) <= 8 * 2.0 ** -24 * np.abs(ref))


def test_bitlinear_rmsnorm_is_scale_invariant(oracle_mod):
    # the normed BitLinear ignores the scale of its input (powers of two,
    # bit for bit), where the plain BitLinear scales with it
    rng = np.random.default_rng(9)
    N, K = 64, 512
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    packed, beta, _ = oracle_mod.pack_weights(W)
    x = (rng.standard_normal((3, K)) * 20).astype(np.float32)
    x[2] = 0.0  # a zero token: h = 0, scale 1e-8, y = 0
    g = (1.0 + 0.1 * rng.standard_normal(K)).astype(np.float32)
    y, acc, xq, s, h, ms = oracle_mod.bitlinear_rmsnorm(x, g, packed, beta, N, K)
    y2, acc2, xq2, s2, _, _ = oracle_mod.bitlinear_rmsnorm(x * np.float32(8.0), g, packed, beta, N, K)
    assert np.array_equal(xq, xq2) and np.array_equal(acc, acc2) and np.array_equal(y, y2)
    assert np.all(xq[2] == 0) and np.all(y[2] == 0.0) and s[2] == np.float32(1e-8)
    # and it is the plain BitLinear of the normed activations
    yb, accb, xqb, sb = oracle_mod.bitlinear(h, packed, beta, N, K)
    assert np.array_equal(y, yb) and np.array_equal(xq, xqb)
