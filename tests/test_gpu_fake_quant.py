"""The training-time (fake-quant) BitLinear forward on the GPU against the
oracle: shadow weights ternarised on each call (packed bytes and beta bit for
bit), the exact int32 products, and y within 1e-6 relative (beta) or within
the one-group bound 9 * 2^-24 * |y| (a learned per-output weight_scale,
y = fl(fl(acc * w_n) * fl(s / 127)))."""
import numpy as np
import pytest

from test_gpu_parity import assert_y_close, to_dev
from ternary_weight_05_b300 import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("learned", [False, True])
@pytest.mark.parametrize("M,N,K", [(1, 300, 2560), (2, 129, 1024), (7, 257, 6912), (300, 200, 2560), (3, 40, 100)])
def test_fake_quant_forward_vs_oracle(lib, oracle_mod, cuda_dev, learned, M, N, K):
    import torch

    rng = np.random.default_rng(M + N + K)
    W = (rng.standard_normal((N, K)) / np.sqrt(K)).astype(np.float32)
    bits, xf = synth.acts_np(M, K, "normal", seed=M * 3 + K, outlier_p=0.001)
    ws = (rng.standard_normal(N) * 0.5 + 1.0).astype(np.float32) if learned else None
    x = to_dev(bits, cuda_dev, torch.bfloat16)
    y, acc, packed, beta = lib.bitlinear_fake_quant(to_dev(W, cuda_dev), x,
                                                    to_dev(ws, cuda_dev) if learned else None,
                                                    want_acc=True, want_packed=True)
    y_ref, cond, acc_ref, _, _, p_ref, b_ref = oracle_mod.bitlinear_fake_quant(W, xf, ws, threads=8)
    assert np.array_equal(packed.cpu().numpy().ravel(), p_ref)
    assert beta.item() == float(b_ref)
    assert np.array_equal(acc.cpu().numpy(), acc_ref)
    if learned:
        err = np.abs(y.cpu().numpy().astype(np.float64) - y_ref)
        assert np.all(err <= 9 * 2.0 ** -24 * cond + 1e-30)
    else:
        assert_y_close(y.cpu().numpy(), y_ref)
    lib.check_device_error()


def test_fake_quant_tracks_weight_updates(lib, oracle_mod, cuda_dev):
    """Two calls with the shadow weights changed in between (a training
    step) use the new ternarisation each time; the workspace is reused."""
    import torch

    N, K = 256, 1024
    rng = np.random.default_rng(5)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    bits, xf = synth.acts_np(1, K, "normal", seed=6)
    x = to_dev(bits, cuda_dev, torch.bfloat16)
    Wd = to_dev(W, cuda_dev)
    ws = torch.zeros(lib.bitlinear_fake_quant_workspace_bytes(1, N, K), dtype=torch.uint8, device=cuda_dev)
    for step in range(3):
        y = lib.bitlinear_fake_quant(Wd, x, workspace=ws)
        y_ref, *_ = oracle_mod.bitlinear_fake_quant(W, xf)
        assert_y_close(y.cpu().numpy(), y_ref)
        W = W - (0.01 * rng.standard_normal((N, K))).astype(np.float32)
        Wd.copy_(torch.from_numpy(W))
