"""bitnet_w2a8_gemv_static_scratch: the decode GEMV for callers that cannot
allocate device memory (a plugin whose host framework owns every device
allocation, a runtime with a fixed, pre-planned memory budget).  It takes its
scratch from a fixed array inside the library instead of a caller workspace.

Checked here through the C ABI: on two calls in a row (the array keeps the
first call's contents) its outputs equal those of bitnet_w2a8_gemv with a
caller workspace and those of the CPU oracle (exact int32 accumulators, fp32
outputs within the 1e-6 relative tolerance of the parity tests); shapes that
need more scratch than the array holds are rejected before anything is
enqueued.

The file name sorts last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest

from ternary_weight_05_b300 import synth

pytestmark = pytest.mark.gpu

RTOL = 1e-6
TOO_LARGE = 8


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _inputs(lib, oracle_mod, dev, M, N, K, seed):
    """Device inputs, and the oracle's outputs on the same weights and
    activations (packed from W and quantised from x on the CPU)."""
    import torch

    W = synth.weights_np(N, K, "normal", 0.02, seed=seed)
    bits, xf = synth.acts_np(M, K, "normal", seed=seed + 1, outlier_p=0.001)
    packed, beta, _ = lib.pack_weights(torch.from_numpy(W).to(dev))
    x = torch.from_numpy(bits).to(dev).view(torch.bfloat16)
    xq, s = lib.quant_act(x)
    p_ref, b_ref, _ = oracle_mod.pack_weights(W)
    y_ref, acc_ref, xq_ref, s_ref = oracle_mod.bitlinear(xf, p_ref, b_ref, N, K, threads=8)
    assert np.array_equal(xq.cpu().numpy(), xq_ref) and np.array_equal(s.cpu().numpy(), s_ref)
    return xq, s, packed, beta, (y_ref, acc_ref)


def _static_call(clib, dev, xq, s, packed, beta, N, K):
    import torch

    M = xq.shape[0]
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
    acc = torch.full((M, N), -7, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    st = clib.bitnet_w2a8_gemv_static_scratch(_ptr(xq), _ptr(s), M, _ptr(packed), _ptr(beta), N, K, _ptr(y),
                                              _ptr(acc), stream)
    assert st == 0, clib.bitnet_status_string(st)
    return y, acc


def _assert_close(y, y_ref):
    y = np.asarray(y, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    zero = y_ref == 0
    assert np.all(y[zero] == 0)
    rel = np.abs(y[~zero] - y_ref[~zero]) / np.abs(y_ref[~zero])
    assert rel.size == 0 or rel.max() <= RTOL, rel.max()


# (M, N, K): M >= 3 runs the stream-K kernel, which uses the scratch (row
# tiles split across CTAs add into it); N is ragged against the 128-row tile.
@pytest.mark.parametrize("M,N,K", [(3, 1000, 2560), (16, 2600, 6912), (64, 13824, 2560), (1, 777, 1024)])
def test_static_scratch_matches_workspace_gemv(lib, oracle_mod, cuda_dev, M, N, K):
    import torch
    from ternary_weight_05_b300 import _lib

    clib = _lib.load()
    assert lib.gemv_workspace_bytes(M, N, K) <= lib.GEMV_STATIC_SCRATCH_BYTES
    for call in range(2):  # two calls in a row: the second sees the first's leftovers
        xq, s, packed, beta, (y_or, acc_or) = _inputs(lib, oracle_mod, cuda_dev, M, N, K,
                                                      seed=1000 * M + 17 * call)
        ws = torch.zeros(lib.gemv_workspace_bytes(M, N, K), dtype=torch.uint8, device=cuda_dev)
        y_ref, acc_ref = lib.w2a8_gemv(xq, s, packed, beta, N, K, want_acc=True, workspace=ws)
        y, acc = _static_call(clib, cuda_dev, xq, s, packed, beta, N, K)
        torch.cuda.synchronize(cuda_dev)
        # against the entry point with a caller workspace
        assert np.array_equal(acc.cpu().numpy(), acc_ref.cpu().numpy()), call
        _assert_close(y.cpu().numpy(), y_ref.cpu().numpy())
        # against the oracle
        assert np.array_equal(acc.cpu().numpy(), acc_or), call
        _assert_close(y.cpu().numpy(), y_or)
    lib.check_device_error()


def test_static_scratch_rejects_oversize(lib, cuda_dev):
    import torch
    from ternary_weight_05_b300 import _lib

    clib = _lib.load()
    M, N, K = 64, 28672, 8192
    assert lib.gemv_workspace_bytes(M, N, K) > lib.GEMV_STATIC_SCRATCH_BYTES
    small = torch.zeros(64, dtype=torch.float32, device=cuda_dev)  # never read: the call is rejected first
    st = clib.bitnet_w2a8_gemv_static_scratch(_ptr(small), _ptr(small), M, _ptr(small), _ptr(small), N, K,
                                              _ptr(small), None, torch.cuda.current_stream(cuda_dev).cuda_stream)
    assert st == TOO_LARGE
    assert clib.bitnet_status_string(st) == b"BITNET_ERR_TOO_LARGE"
    xq = torch.zeros((M, 16), dtype=torch.int8, device=cuda_dev)
    with pytest.raises(_lib.BitnetError):
        lib.w2a8_gemv_static_scratch(xq, small, small, small, N, K)
