"""Failure detection without a fault: a kernel's bounded on-chip wait that
nothing completes gives up after its limit, the device error word reports
BITNET_ERR_TIMEOUT to the host, the word is cleared by the check, and the
context keeps running kernels (a GEMV right after matches the oracle)."""
import numpy as np
import pytest

from test_gpu_parity import assert_y_close, to_dev

pytestmark = pytest.mark.gpu

TIMEOUT = 6


def test_expired_wait_is_reported_and_the_context_survives(lib, oracle_mod, cuda_dev):
    lib.check_device_error()  # nothing pending
    lib.selftest_wait_timeout(2_000_000)  # 2 ms
    with pytest.raises(lib.BitnetError) as err:
        lib.check_device_error()
    assert err.value.status == TIMEOUT
    lib.check_device_error()  # the check cleared the word

    rng = np.random.default_rng(4)
    N, K = 300, 2560
    packed = oracle_mod.pack_codes(rng.integers(-1, 2, size=(N, K)).astype(np.int8))
    xq = rng.integers(-127, 128, size=(1, K)).astype(np.int8)
    s = np.array([1.5], dtype=np.float32)
    y, acc = lib.w2a8_gemv(to_dev(xq, cuda_dev), to_dev(s, cuda_dev), to_dev(packed, cuda_dev),
                           to_dev(np.array([0.5], np.float32), cuda_dev), N, K, want_acc=True)
    acc_ref = oracle_mod.contract(xq, packed, N, K)
    assert np.array_equal(acc.cpu().numpy(), acc_ref)
    assert_y_close(y.cpu().numpy(), oracle_mod.epilogue(acc_ref, s, 0.5))
    lib.check_device_error()


def test_expired_wait_inside_a_pdl_chain(lib, cuda_dev):
    """The self-test kernel between two launches with programmatic dependent
    launch: the error is reported once and cleared."""
    import torch

    x = torch.randn(1, 2560, device=cuda_dev).to(torch.bfloat16)
    W = torch.randn(512, 2560, device=cuda_dev) * 0.02
    packed, beta, _ = lib.pack_weights(W)
    lib.set_pdl(True)
    try:
        y1 = lib.bitlinear(x, packed, beta, 512, 2560)
        lib.selftest_wait_timeout(1_000_000)
        y2 = lib.bitlinear(x, packed, beta, 512, 2560)
    finally:
        lib.set_pdl(False)
    with pytest.raises(lib.BitnetError) as err:
        lib.check_device_error()
    assert err.value.status == TIMEOUT
    assert torch.equal(y1, y2)
    lib.check_device_error()
