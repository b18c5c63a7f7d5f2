"""The BitLinear feed-forward on the GPU against the oracle: the fused
gate/up SwiGLU call (bitnet_bitlinear_swiglu) element by element, and the
whole feed-forward silu(gate(h)) * up(h) -> down.

Tolerance of the SwiGLU product.  The kernels form y = fl(acc * fl(fl(beta *
s) / 127)) (relative error <= 3u, u = 2^-24, against the exact y), then
fl(fl(yg / fl(1 + expf(-yg))) * yu).  expf is within 2 ulp (4u relative);
the argument error |yg| * 3u enters exp(-yg) as a relative error of
|yg| * 3u; 1 + e, the quotient and the product add u each, and the
sensitivity of yg / (1 + e) to e is e / (1 + e) <= 1.  With the 3u of each
y the relative error is at most (13 + 3 |yg|) u; the test allows
(16 + 4 |yg|) u.  Very negative yg (below about -88) make expf overflow and
the fp32 result -0 where the exact value is a tiny subnormal: absolute
tolerance 1e-30 covers that.  The int8 activations, scales and int32
products are compared bit for bit."""
import numpy as np
import pytest

from test_gpu_parity import to_dev
from ternary_weight_05_b300 import synth

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


def assert_swiglu_close(a, a_ref, acc_g, scale, beta_g):
    a = np.asarray(a, dtype=np.float64)
    yg = np.abs(acc_g.astype(np.float64) * beta_g * scale.astype(np.float64)[:, None] / 127.0)
    tol = (16.0 + 4.0 * yg) * U * np.abs(a_ref) + 1e-30
    err = np.abs(a - a_ref)
    bad = err > tol
    assert not bad.any(), (int(bad.sum()), float((err / np.maximum(tol, 1e-300)).max()))


def make_matrices(lib, oracle_mod, dev, I, K, seed, fused_matrix):
    """Gate and up weights, packed on the GPU and by the oracle: two matrices
    with their own beta, or one [2I, K] gate+up matrix (one beta) split into
    its two row halves."""
    if fused_matrix:
        W = synth.weights_np(2 * I, K, "normal", 0.02, seed=seed)
        packed, beta, _ = lib.pack_weights(to_dev(W, dev))
        p_ref, b_ref, _ = oracle_mod.pack_weights(W)
        h = I * K // 4  # the oracle's packed bytes are flat: gate rows, then up rows
        return (packed[:I], beta, packed[I:], beta), (p_ref[:h], b_ref, p_ref[h:], b_ref)
    Wg = synth.weights_np(I, K, "normal", 0.02, seed=seed)
    Wu = synth.weights_np(I, K, "laplace", 0.01, seed=seed + 7)
    pg, bg, _ = lib.pack_weights(to_dev(Wg, dev))
    pu, bu, _ = lib.pack_weights(to_dev(Wu, dev))
    pg_ref, bg_ref, _ = oracle_mod.pack_weights(Wg)
    pu_ref, bu_ref, _ = oracle_mod.pack_weights(Wu)
    return (pg, bg, pu, bu), (pg_ref, bg_ref, pu_ref, bu_ref)


def run_swiglu(lib, oracle_mod, dev, M, I, K, dtype, seed, fused_matrix=False, zero_row=False):
    import torch

    (pg, bg, pu, bu), (pg_ref, bg_ref, pu_ref, bu_ref) = make_matrices(lib, oracle_mod, dev, I, K, seed, fused_matrix)
    bits, xf = synth.acts_np(M, K, "normal", seed=seed + 1, outlier_p=0.001, bf16=(dtype == "bf16"))
    if zero_row and M > 1:
        xf[M - 1] = 0.0
        if bits is not None:
            bits[M - 1] = 0
    x = to_dev(bits, dev, torch.bfloat16) if dtype == "bf16" else to_dev(xf, dev)
    a, acc_g, acc_u, xq, s = lib.bitlinear_swiglu(x, pg, bg, pu, bu, I, K, want_acc=True, want_xq=True)
    a_ref, accg_ref, accu_ref, xq_ref, s_ref = oracle_mod.bitlinear_swiglu(xf, pg_ref, bg_ref, pu_ref, bu_ref, I, K,
                                                                           threads=8)
    s_h = s.cpu().numpy()
    assert np.array_equal(s_h, s_ref)
    assert np.array_equal(xq.cpu().numpy(), xq_ref)
    accg_h = acc_g.cpu().numpy()
    assert np.array_equal(accg_h, accg_ref)
    assert np.array_equal(acc_u.cpu().numpy(), accu_ref)
    assert_swiglu_close(a.cpu().numpy(), a_ref, accg_h, s_h, float(bg.cpu().numpy()[0]))
    lib.check_device_error()
    return a, dict(a=a_ref, acc_g=accg_ref, s=s_ref, beta_g=bg_ref)


# M <= 2: the streaming kernel with silu(gate) * up in its epilogue (row
# lengths 1024..8192 bytes of x, ragged I); M > 2: gate BitLinear + up GEMV /
# GEMM + elementwise product
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("M", [1, 2, 3, 16, 64, 65, 260])
@pytest.mark.parametrize("I,K", [(300, 2560), (129, 1024), (1000, 4096)])
def test_swiglu_vs_oracle(lib, oracle_mod, cuda_dev, dtype, M, I, K):
    run_swiglu(lib, oracle_mod, cuda_dev, M, I, K, dtype, seed=M * 13 + I + K, zero_row=True)


@pytest.mark.parametrize("M,I,K", [(1, 6912, 2560), (2, 6912, 2560), (1, 777, 8192), (4, 6912, 2560)])
def test_swiglu_fused_gate_up_matrix(lib, oracle_mod, cuda_dev, M, I, K):
    run_swiglu(lib, oracle_mod, cuda_dev, M, I, K, "bf16", seed=I + M, fused_matrix=True)


# shapes the streaming kernel does not take (K % 64 != 0, K < 512, K too long)
@pytest.mark.parametrize("M,I,K", [(1, 50, 100), (2, 70, 448), (1, 33, 16384), (2, 40, 8192)])
def test_swiglu_other_shapes(lib, oracle_mod, cuda_dev, M, I, K):
    run_swiglu(lib, oracle_mod, cuda_dev, M, I, K, "bf16", seed=M + I + K)


def test_swiglu_epilogue_equals_elementwise_path(lib, oracle_mod, cuda_dev):
    """The fused epilogue and the elementwise kernel give the same bits: x at
    a 2-byte offset is not 16-byte aligned, which sends the same problem down
    the gate BitLinear + up GEMV + elementwise path."""
    import torch

    M, I, K = 2, 2000, 2560
    (pg, bg, pu, bu), _ = make_matrices(lib, oracle_mod, cuda_dev, I, K, 5, False)
    bits, _ = synth.acts_np(M, K, "normal", seed=6)
    x = to_dev(bits, cuda_dev, torch.bfloat16)
    buf = torch.empty(M * K + 8, dtype=torch.bfloat16, device=cuda_dev)
    x_off = buf[1:1 + M * K].view(M, K)
    x_off.copy_(x)
    assert x_off.data_ptr() % 16 != 0
    a1 = lib.bitlinear_swiglu(x, pg, bg, pu, bu, I, K)
    a2 = lib.bitlinear_swiglu(x_off, pg, bg, pu, bu, I, K)
    assert np.array_equal(a1.cpu().numpy().view(np.uint32), a2.cpu().numpy().view(np.uint32))


def down_reference(oracle_mod, ref, pd_ref, bd_ref, D, I):
    """The oracle's down BitLinear on fl32 of its exact SwiGLU product, the
    bound `rel` on the relative error of each row of the GPU's product (the
    product's bound plus the rounding to fp32) and the positions `near` where
    a / s * 127 lies within that error of a rounding midpoint."""
    a32 = ref["a"].astype(np.float32)
    y_ref, acc_ref, xq_ref, s_ref = oracle_mod.bitlinear(a32, pd_ref, bd_ref, D, I, threads=8)
    yg = np.abs(ref["acc_g"].astype(np.float64) * ref["beta_g"] * ref["s"].astype(np.float64)[:, None] / 127.0)
    rel = ((16.0 + 4.0 * yg) * U).max(axis=1) + U
    s64 = s_ref.astype(np.float64)
    t = np.abs(a32.astype(np.float64)) / s64[:, None] * 127.0
    near = np.abs(t - np.floor(t) - 0.5) <= (2.0 * rel[:, None] + 4.0 * U) * np.maximum(t, 1.0)
    return dict(y=y_ref, acc=acc_ref, xq=xq_ref, s=s_ref, rel=rel, near=near, beta=float(bd_ref))


def assert_down_close(y, dref, flips):
    """y within the usual tolerance plus twice the scale's relative error,
    plus `flips` (per row) steps of w_scale * s / 127."""
    from test_gpu_parity import RTOL

    step = dref["beta"] * dref["s"].astype(np.float64) / 127.0
    y64, yr64 = np.asarray(y, dtype=np.float64), dref["y"].astype(np.float64)
    tol = (RTOL + 2.0 * dref["rel"][:, None]) * np.abs(yr64) + flips[:, None] * step[:, None] * (1.0 + 1e-6)
    assert np.all(np.abs(y64 - yr64) <= tol)


@pytest.mark.parametrize("M,D,I", [(1, 2560, 6912), (2, 1024, 2048), (16, 1024, 2048)])
def test_ffn_vs_oracle(lib, oracle_mod, cuda_dev, M, D, I):
    """silu(gate(h)) * up(h) -> down, the feed-forward of the BitTransformer
    block, against the oracle run on the same h.  The down BitLinear quantises
    the fp32 product a; the oracle quantises fl32 of its exact a.  Where
    a / s * 127 lies within the product's error bound of a rounding midpoint
    the two may round apart by one step: such positions are found from the
    oracle's values; the GPU's int8 activations must equal the oracle's
    everywhere else and be within one step there, each down accumulator may
    differ by at most the number of such steps in its row, and y by that many
    steps of w_scale * s / 127 beyond the usual tolerance and the scale's
    relative error."""
    a, ref = run_swiglu(lib, oracle_mod, cuda_dev, M, I, D, "bf16", seed=D + I + M)
    Wd = synth.weights_np(D, I, "normal", 0.02, seed=77)
    pd, bd, _ = lib.pack_weights(to_dev(Wd, cuda_dev))
    pd_ref, bd_ref, _ = oracle_mod.pack_weights(Wd)
    y, acc, xq, s = lib.bitlinear(a, pd, bd, D, I, want_acc=True, want_xq=True)
    dref = down_reference(oracle_mod, ref, pd_ref, bd_ref, D, I)

    s_h, xq_h, acc_h = s.cpu().numpy(), xq.cpu().numpy(), acc.cpu().numpy()
    s64 = dref["s"].astype(np.float64)
    # the scale is max |a|: within the bound of the element that attains it
    assert np.all(np.abs(s_h.astype(np.float64) - s64) <= dref["rel"] * s64)
    diff = xq_h.astype(np.int32) - dref["xq"].astype(np.int32)
    assert np.all(diff[~dref["near"]] == 0)
    assert np.all(np.abs(diff) <= 1)
    flips = np.abs(diff).sum(axis=1)
    assert np.all(np.abs(acc_h.astype(np.int64) - dref["acc"]) <= flips[:, None])
    if not flips.any():
        assert np.array_equal(acc_h, dref["acc"])
    assert_down_close(y.cpu().numpy(), dref, flips)
    lib.check_device_error()
