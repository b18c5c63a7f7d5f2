"""RMSNorm in front of the BitLinear (bitnet_rmsnorm_quant_act and
bitnet_bitlinear_rmsnorm) against the oracle, element by element.

The mean square ms = fl32(S / K) comes from an fp64 sum of squares whose
order is the kernel's own; the oracle sums left to right.  Both sums are
within (K - 1) * 2^-53 * S of the exact S, so the two ms can differ only
where S / K lies within 2 (K - 1) * 2^-53 * S / K of the midpoint between
two fp32 values.  Where the GPU's ms differs from the oracle's, the test
requires the two to be such neighbours with the exact S / K inside that
window, and then checks every later value against the oracle's arithmetic
carried out with the GPU's ms (oracle.rmsnorm_apply).  Everywhere else: h,
x_q, scales and int32 products bit-exact, y within 1e-6 relative.
"""
import math

import numpy as np
import pytest

from test_gpu_parity import assert_y_close, to_dev
from ternary_weight_05_b300 import synth

pytestmark = pytest.mark.gpu

EPS = 2.0 ** -23


def reference(oracle_mod, xf, g, ms_gpu, eps=EPS):
    """The oracle's h per token, with the GPU's mean square where the two
    differ inside the window of an fp32 rounding boundary."""
    h, ms = oracle_mod.rmsnorm(xf, g, eps)
    M, K = xf.shape
    for m in np.nonzero(ms_gpu != ms)[0]:
        a, b = sorted((float(ms[m]), float(ms_gpu[m])))
        assert np.nextafter(np.float32(a), np.float32(np.inf)) == np.float32(b), (m, a, b)
        S = math.fsum(float(v) * float(v) for v in xf[m].astype(np.float64))
        mid = (a + b) / 2.0
        assert abs(S / K - mid) <= (2 * K * 2.0 ** -53 + 2.0 ** -52) * (S / K), (m, S / K, mid)
        h[m], _ = oracle_mod.rmsnorm_apply(xf[m], ms_gpu[m], g, eps)
    return h


def inputs(M, K, dtype, seed, scale=1.0):
    bits, xf = synth.acts_np(M, K, "student_t4", seed=seed, outlier_p=0.002, bf16=(dtype == "bf16"))
    if scale != 1.0:
        xf = (xf * np.float32(scale)).astype(np.float32)
        if bits is not None:
            bits = synth.f32_to_bf16_bits(xf)
            xf = synth.bf16_bits_to_f32(bits)
    if M > 2:
        xf[1] = 0.0
        if bits is not None:
            bits[1] = 0
    return bits, xf


def device_x(bits, xf, dev):
    import torch

    return to_dev(bits, dev, torch.bfloat16) if bits is not None else to_dev(xf, dev)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("weighted", [False, True])
@pytest.mark.parametrize("M,K,scale", [(1, 8192, 1.0), (3, 2560, 1e-3), (5, 6912, 300.0), (64, 1000, 1.0),
                                       (2, 8, 1.0), (17, 12288, 2.0 ** -60)])
def test_rmsnorm_quant_act(lib, oracle_mod, cuda_dev, dtype, weighted, M, K, scale):
    bits, xf = inputs(M, K, dtype, seed=M * 7 + K, scale=scale)
    g = (np.random.default_rng(K).standard_normal(K) * 0.5 + 1.0).astype(np.float32) if weighted else None
    gd = to_dev(g, cuda_dev) if weighted else None
    xq, s, h, ms = lib.rmsnorm_quant_act(device_x(bits, xf, cuda_dev), gd, want_h=True, want_ms=True)
    ms_g = ms.cpu().numpy()
    h_ref = reference(oracle_mod, xf, g, ms_g)
    assert np.array_equal(h.cpu().numpy().view(np.uint32), h_ref.view(np.uint32))
    xq_ref, s_ref = oracle_mod.quant_act(h_ref)
    assert np.array_equal(s.cpu().numpy(), s_ref)
    assert np.array_equal(xq.cpu().numpy(), xq_ref)


# M <= 2: rmsnorm_quant_act + the streaming GEMV; 3..64: the prep kernel with
# the RMSNorm + tensor-core GEMV; > 64: the same prep + tcgen05 GEMM; K % 64
# != 0: the unfused route for every M
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("M", [1, 2, 3, 16, 64, 65, 300])
@pytest.mark.parametrize("N,K", [(300, 2560), (257, 8192), (129, 1000)])
def test_bitlinear_rmsnorm(lib, oracle_mod, cuda_dev, dtype, M, N, K):
    import torch

    bits, xf = inputs(M, K, dtype, seed=M * 31 + N + K)
    g = (np.random.default_rng(N).standard_normal(K) * 0.3 + 1.0).astype(np.float32)
    W = synth.weights_np(N, K, "normal", 0.02, seed=M + N)
    packed, beta, _ = lib.pack_weights(to_dev(W, cuda_dev))
    p_ref, b_ref, _ = oracle_mod.pack_weights(W)
    ws = torch.empty(lib.bitlinear_workspace_bytes(M, N, K), dtype=torch.uint8, device=cuda_dev)
    ws.fill_(0x3C)  # any contents
    y, acc, xq, s, ms = lib.bitlinear_rmsnorm(device_x(bits, xf, cuda_dev), to_dev(g, cuda_dev), packed, beta, N, K,
                                              want_acc=True, want_xq=True, want_ms=True, workspace=ws)
    h_ref = reference(oracle_mod, xf, g, ms.cpu().numpy())
    y_ref, acc_ref, xq_ref, s_ref = oracle_mod.bitlinear(h_ref, p_ref, b_ref, N, K, threads=8)
    assert np.array_equal(s.cpu().numpy(), s_ref)
    assert np.array_equal(xq.cpu().numpy(), xq_ref)
    assert np.array_equal(acc.cpu().numpy(), acc_ref)
    assert_y_close(y.cpu().numpy(), y_ref)
    # the same products through the standalone norm + the int8 matmul
    xq2, s2 = lib.rmsnorm_quant_act(device_x(bits, xf, cuda_dev), to_dev(g, cuda_dev))
    f = lib.w2a8_gemv if M <= lib.GEMV_MAX_M else lib.w2a8_gemm
    y2 = f(xq2, s2, packed, beta, N, K)
    assert np.array_equal(y.cpu().numpy().view(np.uint32), y2.cpu().numpy().view(np.uint32))
    lib.check_device_error()
