"""The fused BitLinear forward (bitnet_bitlinear: absmax quantisation inside
the matmul kernels) against the oracle, element by element: bit-exact x_q,
scales and int32 accumulators, fp32 outputs within 1e-6 relative; and
bitwise equal to the unfused quant_act -> GEMV / GEMM sequence."""
import numpy as np
import pytest

from test_gpu_parity import assert_y_close, to_dev
from ternary_weight_05_b300 import synth

pytestmark = pytest.mark.gpu


def run_case(lib, oracle_mod, dev, M, N, K, dtype, seed, zero_row=False, dist="student_t4"):
    import torch

    W = synth.weights_np(N, K, "normal", 0.02, seed=seed)
    bits, xf = synth.acts_np(M, K, dist, seed=seed + 1, outlier_p=0.002, bf16=(dtype == "bf16"))
    if zero_row and M > 1:
        xf[M // 2] = 0.0
        if bits is not None:
            bits[M // 2] = 0
    x = to_dev(bits, dev, torch.bfloat16) if dtype == "bf16" else to_dev(xf, dev)
    packed, beta, _ = lib.pack_weights(to_dev(W, dev))
    y, acc, xq, s = lib.bitlinear(x, packed, beta, N, K, want_acc=True, want_xq=True)
    p_ref, b_ref, _ = oracle_mod.pack_weights(W)
    y_ref, acc_ref, xq_ref, s_ref = oracle_mod.bitlinear(xf, p_ref, b_ref, N, K, threads=8)
    assert np.array_equal(s.cpu().numpy(), s_ref)
    assert np.array_equal(xq.cpu().numpy(), xq_ref)
    assert np.array_equal(acc.cpu().numpy(), acc_ref)
    assert_y_close(y.cpu().numpy(), y_ref)
    # the unfused calls give the same bits
    xq2, s2 = lib.quant_act(x)
    f = lib.w2a8_gemv if M <= lib.GEMV_MAX_M else lib.w2a8_gemm
    y2 = f(xq2, s2, packed, beta, N, K)
    assert np.array_equal(y.cpu().numpy().view(np.uint32), y2.cpu().numpy().view(np.uint32))
    return y


# fused streaming kernel (M <= 2), fused prep + mma.sync GEMV (3..64), fused
# prep + tcgen05 GEMM (> 64); ragged N, K not a multiple of 512
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("M", [1, 2, 3, 16, 64, 65, 300])
# K = 8192: the streaming kernel's full-register edge for one token (four
# 16-byte chunks per lane) and the row-range kernel for two; ragged N
@pytest.mark.parametrize("N,K", [(300, 2560), (129, 1024), (257, 6912), (777, 8192), (4097, 8192)])
def test_bitlinear_fused(lib, oracle_mod, cuda_dev, dtype, M, N, K):
    run_case(lib, oracle_mod, cuda_dev, M, N, K, dtype, seed=M * 31 + N + K, zero_row=True)


# shapes the fused kernels do not take: quant_act + matmul entry points
@pytest.mark.parametrize("M,N,K", [(1, 40, 100), (5, 33, 448), (70, 20, 96), (3, 40, 66048)])
def test_bitlinear_unfused_shapes(lib, oracle_mod, cuda_dev, M, N, K):
    run_case(lib, oracle_mod, cuda_dev, M, N, K, "bf16", seed=M + N + K, dist="normal")


def test_bitlinear_workspace_reuse_and_outputs_optional(lib, oracle_mod, cuda_dev):
    import torch

    N, K = 1000, 2560
    W = synth.weights_np(N, K, "normal", 0.02, seed=9)
    packed, beta, _ = lib.pack_weights(to_dev(W, cuda_dev))
    p_ref, b_ref, _ = oracle_mod.pack_weights(W)
    ws = torch.zeros(max(lib.bitlinear_workspace_bytes(M, N, K) for M in (1, 8, 40)), dtype=torch.uint8,
                     device=cuda_dev)
    for rep in range(2):
        for M in (1, 8, 40):
            bits, xf = synth.acts_np(M, K, "normal", seed=100 * rep + M)
            y = lib.bitlinear(to_dev(bits, cuda_dev, torch.bfloat16), packed, beta, N, K, workspace=ws)
            y_ref, _, _, _ = oracle_mod.bitlinear(xf, p_ref, b_ref, N, K, threads=8)
            assert_y_close(y.cpu().numpy(), y_ref)
    lib.check_device_error()


# Two tokens with rows longer than 4096 on a matrix of at least 2^27 weights
# run on the tensor-core GEMV instead of the row-range kernel; N is ragged
# against the 128-row tile.
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_bitlinear_two_tokens_large_matrix(lib, oracle_mod, cuda_dev, dtype):
    N, K = 16389, 8192
    assert N * K >= 1 << 27
    run_case(lib, oracle_mod, cuda_dev, 2, N, K, dtype, seed=77, zero_row=False)
